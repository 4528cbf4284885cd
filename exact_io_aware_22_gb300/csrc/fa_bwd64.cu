// fa_bwd64.cu -- attention backward (dK/dV and dQ) on sm_103a for head dims 32 and
// 64, as persistent kernels (the pre-pass is in fa_bwd.cu; d = 128 runs the kernels of
// fa_bwd128.cu).
//
// Method: "flash-attn-triton" docs page, section "Scope" (backward kernels for
// dQ, dK, dV that rebuild P from the saved L; causal mask only on diagonal
// tiles; ragged N) and "Source" (delta pre-pass, then dK/dV, then dQ).
// Gradients follow the chain rule of the forward:
//   P = exp(S - L),  dV = P^T dO,  dP = dO V^T,  D = rowsum(dO o O),
//   dS = P o (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
//
// At these head dims a work item (one 128-key block in dK/dV, one 128-query tile
// in dQ) holds few tiles of work, and a CTA per item spent as long on its set-up,
// first loads, pipeline refill and stores as on its products.  Here one CTA per SM
// runs from item to item: it starts with the item of its own index and takes further
// items from CTAs that have not been launched yet (cluster launch control), so the
// grid's longest-first order still decides what comes next.  An item's K/V (dK/dV)
// or Q/dO (dQ) tiles are double-buffered in shared memory so its loads overlap the
// previous item, and results leave through shared memory as coalesced rows.  The
// head dim leaves room in TMEM for every intermediate of a tile to have columns of
// its own, so no product waits for another product's operand to be consumed.
//
// Roles (640 threads, one CTA per SM):
//   warp 0       TMA producer and scheduler: publishes each item in a two-slot ring,
//                streams its tiles, then asks for the next item.
//   warp 1       TMEM allocator; lane 0 issues the score MMAs (dK/dV: S^T, dP^T; dQ:
//                S, dP).
//   warp 2       lane 0 issues the gradient MMAs (dK/dV: dV, dK; dQ: dQ).
//   warp 3       idle; it completes the first warpgroup for the register split.
//   warps 4-19   four compute warpgroups, one thread per TMEM lane (a key row in dK/dV,
//                a query row in dQ) and 32 columns of each 128-column score tile.  The
//                element-wise work of a tile (exponentials, dS) is the same at every head
//                dim, while the products shrink with it; at d <= 64 a tile's compute,
//                not its MMAs, set the pace with two warps per scheduler, so the tile is
//                cut four ways.  The producer / MMA warpgroup hands registers to the
//                compute warpgroups (setmaxnreg: 56 and 104 of the 96 per thread given
//                at launch).
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
constexpr int THREADS = 640;
constexpr uint32_t kRegs64Launch = 96, kRegs64Low = 56, kRegs64High = 104;
static_assert(128 * kRegs64Low + 512 * kRegs64High <= THREADS * kRegs64Launch,
              "register split must fit the launch allocation");

// Rows of one warp's 32 TMEM lanes, NC (32) fp32 columns from taddr times mul, rounded to
// the 16-bit type, written to global memory through this warp's 32 staging rows in
// shared memory (row r's 16-byte chunk c at chunk c ^ (r mod 4), so the lanes of a
// store phase hit distinct banks): each store instruction then writes eight rows of 64
// contiguous bytes.  row_ptr(r) is where row r's NC values go; rows r >= n_valid are
// not written.
template <bool BF16, typename RowPtr>
__device__ __forceinline__ void store_rows_staged(uint32_t taddr, float mul, uint4* stage,
                                                  int lane, RowPtr row_ptr, int n_valid) {
  constexpr int CPR = 4;                         // 16-byte chunks per 32-column row
  uint32_t v[32];
  tmem_ld32(taddr, v);
  tmem_ld_wait_regs(v);
#pragma unroll
  for (int i = 0; i < CPR; ++i) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = pack2<BF16>(__uint_as_float(v[8 * i + 2 * e]) * mul,
                         __uint_as_float(v[8 * i + 2 * e + 1]) * mul);
    stage[lane * CPR + (i ^ (lane % CPR))] = make_uint4(w[0], w[1], w[2], w[3]);
  }
  __syncwarp();
  constexpr int RPI = 32 / CPR;                  // rows per store instruction
#pragma unroll
  for (int i = 0; i < 32 / RPI; ++i) {
    const int r = i * RPI + lane / CPR, c = lane % CPR;
    if (r < n_valid) *(reinterpret_cast<uint4*>(row_ptr(r)) + c) = stage[r * CPR + (c ^ (r % CPR))];
  }
  __syncwarp();
}

// ============================================================== dK / dV
namespace kv64 {
// K and V of two work items; Q with L*log2e in a 3-stage ring, dO with D in a 2-stage
// ring (both rings run on across items); dV and dK rows staged for the store.
template <int HD>
struct Smem {
  static constexpr int TILE = BT * HD * 2;
  static constexpr int Q_STAGES = 3, DO_STAGES = 2;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = 2 * TILE;
  static constexpr int Q_OFF = 4 * TILE;
  static constexpr int DO_OFF = Q_OFF + Q_STAGES * TILE;
  static constexpr int L_OFF = DO_OFF + DO_STAGES * TILE;   // per Q stage: 128 L*log2e
  static constexpr int D_OFF = L_OFF + Q_STAGES * 512;      // per dO stage: 128 D
  static constexpr int ST_OFF = D_OFF + DO_STAGES * 512;    // 32-column row slices, 8 KiB
  static constexpr int BAR_OFF = ST_OFF + 4 * 8192;          // per compute warpgroup
  // kv_full[2], kv_empty[2], q_full[3], q_empty[3], do_full[2], do_empty[2], s_full, s_free,
  // dp_full, dp_free, p_ready, p_free, ds_ready, ds_free, out_full, acc_free, done[2],
  // tile_full[2], tile_empty[2], clc
  static constexpr int NBARS = 4 + 2 * Q_STAGES + 2 * DO_STAGES + 8 + 2 + 2 + 4 + 1;
  static constexpr int CLC_OFF = (BAR_OFF + NBARS * 8 + 15) / 16 * 16;   // 16-byte response
  static constexpr int SLOT_OFF = CLC_OFF + 16;             // TMEM base, item slots[2]
  static constexpr int SMEM_BYTES = SLOT_OFF + 16;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA exceeds 227 KiB");
};
// TMEM: dV | dK (HD of 64 columns each) | S^T (128) | dP^T (128) | P^T | dS^T (64 each,
// 16-bit pairs).  Compute warpgroup q owns query columns [32q, 32q + 32) of S^T and
// dP^T, and pair columns [16q, 16q + 16) of P^T and dS^T, the A operands of
// dV += P^T dO and dK += dS^T Q.  Pipe order per tile i: S^T(i+1), dP^T(i+1), dV(i),
// dK(i); S^T and dP^T of the next tile are issued as soon as the compute warps have
// read this tile's, P^T and dS^T are written once the previous tile's dV and dK have
// read theirs.
constexpr uint32_t DV_COL = 0, DK_COL = 64, S_COL = 128, DP_COL = 256, P_COL = 384,
                   DS_COL = 448;

// One key block of one K/V head and the query tiles that see it.
struct Item {
  int bkv, kb, hk, q_start, n_head, n_iter;
  SeqRows sr;
};
template <bool CAUSAL>
__device__ __forceinline__ Item item(int id, int nkb, int ord_g, int N, int group, int window,
                                     const int* __restrict__ cu_seqlens, int H, int total) {
  Item t;
  const BlockPos bp = block_pos(nkb, id, ord_g);
  t.bkv = bp.bh;                                  // K/V head; its query heads: bkv*group + g
  t.kb = bp.rank;                                 // causal: block 0 has the most work
  t.q_start = CAUSAL ? t.kb : 0;                  // the diagonal query tile
  const int Hkv = H / group;
  t.sr = seq_rows(cu_seqlens, t.bkv / Hkv, N, total);
  t.hk = t.sr.packed ? t.bkv % Hkv : t.bkv;
  const int nq_r = (t.sr.n + BT - 1) / BT;
  // query tiles per query head: from the diagonal to the last tile that sees a key of
  // this block (with a window of W keys, query rows up to the block's last key + W - 1)
  t.n_head = t.kb * BT >= t.sr.n ? 0
      : ((CAUSAL && window > 0) ? min(nq_r, (t.kb * BT + BT - 1 + window - 1) / BT + 1) : nq_r) -
            t.q_start;
  t.n_iter = t.n_head > 0 ? group * t.n_head : 0;  // the group's query heads one after another
  return t;
}
}  // namespace kv64

template <int HD, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(THREADS, 1)
    dkdv64_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const float* __restrict__ Dp, const float* __restrict__ Lp,
                  void* __restrict__ dK, void* __restrict__ dV, int N, int Np, int group,
                  int window, const int* __restrict__ cu_seqlens, int H, int total, float scale,
                  float c_log2, int ord_g, KernelCtl ctl) {
  using namespace kv64;
  using SM = Smem<HD>;
  using G = Geo<HD>;
  constexpr int TILE = SM::TILE, Q_STAGES = SM::Q_STAGES, DO_STAGES = SM::DO_STAGES;
  extern __shared__ __align__(1024) uint8_t sg[];
  const uint32_t sb = smem_u32(sg);
  grid_dep_launch();
  if (sb & 1023u) {                                // see FA_DEV_SMEM_ALIGN
    grid_dep_wait();
    if (threadIdx.x == 0) atomicOr(ctl.status, FA_DEV_SMEM_ALIGN);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = (N + BT - 1) / BT;
  const int Hkv = H / group;
  auto item_of = [&](int id) {
    return item<CAUSAL>(id, nkb, ord_g, N, group, window, cu_seqlens, H, total);
  };

  auto bar = [&](int i) -> uint32_t { return sb + SM::BAR_OFF + 8 * i; };
  auto B_KVF = [&](int b) { return b; };
  auto B_KVE = [&](int b) { return 2 + b; };
  auto B_QF = [&](int s) { return 4 + s; };
  auto B_QE = [&](int s) { return 4 + Q_STAGES + s; };
  auto B_GF = [&](int g) { return 4 + 2 * Q_STAGES + g; };   // dO and D of a stage
  auto B_GE = [&](int g) { return 4 + 2 * Q_STAGES + DO_STAGES + g; };
  const int B_SF = 4 + 2 * Q_STAGES + 2 * DO_STAGES, B_SFREE = B_SF + 1, B_DPF = B_SF + 2,
            B_DPFREE = B_SF + 3, B_PR = B_SF + 4, B_PFREE = B_SF + 5, B_DR = B_SF + 6,
            B_DSFREE = B_SF + 7, B_OF = B_SF + 8, B_AF = B_SF + 9, B_DONE = B_SF + 10,
            B_DONE2 = B_SF + 11;
  auto B_TF = [&](int b) { return B_SF + 12 + b; };
  auto B_TE = [&](int b) { return B_SF + 14 + b; };
  const int B_CLC = B_SF + 16;
  volatile int* slot = reinterpret_cast<volatile int*>(sg + SM::SLOT_OFF + 4);
  const uint32_t clc_resp = sb + SM::CLC_OFF;

  if (threadIdx.x == 0) {
    for (int i = 0; i < SM::NBARS; ++i) mbar_init(bar(i), 1);
    mbar_init(bar(B_SFREE), 512);
    mbar_init(bar(B_DPFREE), 512);
    mbar_init(bar(B_PR), 512);
    mbar_init(bar(B_DR), 512);
    mbar_init(bar(B_AF), 512);
    for (int i = 0; i < Q_STAGES; ++i) mbar_init(bar(B_QE(i)), 2);   // both MMA issuers
    for (int i = 0; i < DO_STAGES; ++i) mbar_init(bar(B_GE(i)), 2);
    mbar_init(bar(B_TE(0)), 18);                   // the MMA issuers and one lane per compute warp
    mbar_init(bar(B_TE(1)), 18);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sb + SM::SLOT_OFF, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sg + SM::SLOT_OFF);
  grid_dep_wait();                                 // D and L*log2e from the pre-pass

  auto next_item = [&](int k, bool& ok) -> int {
    if (!(ok = mbar_wait(bar(B_TF(k & 1)), (k >> 1) & 1, ctl))) return -1;
    return slot[k & 1];
  };

  if (warp == 0) {
    regs_dec<kRegs64Low>();                        // warpgroup 0 (TMA, MMA issue): few registers
    // ------------------------------------------------------------ producer, scheduler
    if (lane == 0) {
      bool ok = true;
      int id = static_cast<int>(blockIdx.x);
      int gi = 0, kq = 0, nq = 0, ng = 0;         // Q/dO tiles, items, Q and dO loads issued
      bool pending = false;                        // a request for the next item is out
      int n_req = 0;                               // requests made
      for (int k = 0; ok; ++k) {
        if (!(ok = mbar_wait(bar(B_TE(k & 1)), ((k >> 1) & 1) ^ 1, ctl))) break;
        slot[k & 1] = id;
        mbar_arrive(bar(B_TF(k & 1)));
        if (id < 0) break;
        // ask for the next item together with this item's last loads: early enough that
        // the answer is there when they complete, late enough that a CTA takes an item
        // only when it is nearly free
        auto request = [&]() {
          mbar_arrive_expect_tx(bar(B_CLC), 16);
          clc_try_cancel(clc_resp, bar(B_CLC));
          pending = true;
          ++n_req;
        };
        const Item t = item_of(id);
        if (t.n_iter <= 0) request();
        if (t.n_iter > 0) {
          const int kvb = kq & 1;
          if (!(ok = mbar_wait(bar(B_KVE(kvb)), ((kq >> 1) & 1) ^ 1, ctl))) break;
          mbar_arrive_expect_tx(bar(B_KVF(kvb)), 2 * TILE);
          for (int c = 0; c < G::NCH; ++c) {
            tma_load_3d(sb + SM::K_OFF + kvb * TILE + c * G::CHUNK, &tmK, bar(B_KVF(kvb)),
                        c * G::SPAN, t.sr.y(t.kb * BT, t.hk), t.sr.z(t.kb * BT, t.hk));
            tma_load_3d(sb + SM::V_OFF + kvb * TILE + c * G::CHUNK, &tmV, bar(B_KVF(kvb)),
                        c * G::SPAN, t.sr.y(t.kb * BT, t.hk), t.sr.z(t.kb * BT, t.hk));
          }
          ++kq;
          for (int it = 0; it < t.n_iter; ++it, ++gi) {
            const int s = gi % Q_STAGES, g = gi % DO_STAGES;
            const int gh = it / t.n_head;           // which query head of the group
            const int qrow = (t.q_start + it - gh * t.n_head) * BT, bhq = t.bkv * group + gh;
            const int hq = t.sr.packed ? bhq % H : bhq;
            const size_t row = static_cast<size_t>(bhq) * Np + qrow;
            if (!(ok = mbar_wait(bar(B_QE(s)), ((gi / Q_STAGES) & 1) ^ 1, ctl))) break;
            mbar_arrive_expect_tx(bar(B_QF(s)), TILE + 512);
            for (int c = 0; c < G::NCH; ++c)
              tma_load_3d(sb + SM::Q_OFF + s * TILE + c * G::CHUNK, &tmQ, bar(B_QF(s)),
                          c * G::SPAN, t.sr.y(qrow, hq), t.sr.z(qrow, hq));
            bulk_load(sb + SM::L_OFF + s * 512, Lp + row, 512, bar(B_QF(s)));
            ++nq;
            if (!(ok = mbar_wait(bar(B_GE(g)), ((gi / DO_STAGES) & 1) ^ 1, ctl))) break;
            mbar_arrive_expect_tx(bar(B_GF(g)), TILE + 512);
            for (int c = 0; c < G::NCH; ++c)
              tma_load_3d(sb + SM::DO_OFF + g * TILE + c * G::CHUNK, &tmdO, bar(B_GF(g)),
                          c * G::SPAN, t.sr.y(qrow, hq), t.sr.z(qrow, hq));
            bulk_load(sb + SM::D_OFF + g * 512, Dp + row, 512, bar(B_GF(g)));
            ++ng;
            if (it + 1 == t.n_iter) request();
          }
          if (!ok) break;
        }
        // the next item: a CTA that had not started, if any was left
        if (!(ok = mbar_wait(bar(B_CLC), k & 1, ctl))) break;
        pending = false;
        id = clc_result(clc_resp);
      }
      if (!ok) {
        if (pending) mbar_wait(bar(B_CLC), (n_req - 1) & 1, ctl);   // the response lands in smem
        // drain: wait (bounded) for the copies this thread may still have in flight
        for (int i = max(0, kq - 2); i < kq; ++i) mbar_wait(bar(B_KVF(i & 1)), (i >> 1) & 1, ctl);
        for (int i = max(0, nq - Q_STAGES); i < nq; ++i)
          mbar_wait(bar(B_QF(i % Q_STAGES)), (i / Q_STAGES) & 1, ctl);
        for (int i = max(0, ng - DO_STAGES); i < ng; ++i)
          mbar_wait(bar(B_GF(i % DO_STAGES)), (i / DO_STAGES) & 1, ctl);
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    regs_dec<kRegs64Low>();
    // ------------------------------------------------------------ MMA issuers
    // Two threads issue, so the tensor pipe is not held to one thread's issue rate:
    // warp 1 the score products S^T = K Q^T and dP^T = V dO^T, warp 2 the gradient
    // products dV += P^T dO and dK += dS^T Q.  A Q or dO stage is free once both
    // threads' products that read it have completed (those barriers count two commits).
    if (lane == 0) {
      const bool scores = warp == 1;
      constexpr uint32_t idS = umma_idesc_f16(BT, BT, BF16, false, false);   // S^T, dP^T
      constexpr uint32_t idG = umma_idesc_f16(BT, HD, BF16, false, true);    // dV, dK
      constexpr uint32_t HI = G::HI, STAGE_W = TILE >> 4;
      const uint32_t k_lo = sdesc_lo(sb + SM::K_OFF, 16), v_lo = sdesc_lo(sb + SM::V_OFF, 16);
      const uint32_t q_lo = sdesc_lo(sb + SM::Q_OFF, 16), qm_lo = sdesc_lo(sb + SM::Q_OFF, G::CHUNK);
      const uint32_t o_lo = sdesc_lo(sb + SM::DO_OFF, 16), om_lo = sdesc_lo(sb + SM::DO_OFF, G::CHUNK);
      bool ok = true;
      int gi = 0, kq = 0;
      for (int k = 0; ok; ++k) {
        const int id = next_item(k, ok);
        if (!ok) break;
        mbar_arrive(bar(B_TE(k & 1)));
        if (id < 0) break;
        const Item t = item_of(id);
        if (t.n_iter <= 0) continue;
        const int kvb = kq & 1;
        if (scores) {
          const uint32_t ka = k_lo + kvb * STAGE_W, va = v_lo + kvb * STAGE_W;
          if (!(ok = mbar_wait(bar(B_KVF(kvb)), (kq >> 1) & 1, ctl))) break;
          for (int it = 0; ok && it < t.n_iter; ++it, ++gi) {
            // S^T(g) and dP^T(g) once their tiles are in and the compute warps have read
            // the previous tile's
            const int s = gi % Q_STAGES, g = gi % DO_STAGES;
            if (!(ok = mbar_wait(bar(B_QF(s)), (gi / Q_STAGES) & 1, ctl))) break;
            if (gi > 0 && !(ok = mbar_wait(bar(B_SFREE), (gi - 1) & 1, ctl))) break;
            tc_fence_after();
            issue_ab_t_w<HD>(tmem + S_COL, ka, q_lo + s * STAGE_W, idS);
            umma_commit(bar(B_SF));
            if (!(ok = mbar_wait(bar(B_GF(g)), (gi / DO_STAGES) & 1, ctl))) break;
            if (gi > 0 && !(ok = mbar_wait(bar(B_DPFREE), (gi - 1) & 1, ctl))) break;
            tc_fence_after();
            issue_ab_t_w<HD>(tmem + DP_COL, va, o_lo + g * STAGE_W, idS);
            umma_commit(bar(B_DPF));
            umma_commit(bar(B_QE(s)));
            umma_commit(bar(B_GE(g)));
          }
          if (!ok) break;
          umma_commit(bar(B_KVE(kvb)));            // this item's K, V no longer read
        } else {
          for (int it = 0; ok && it < t.n_iter; ++it, ++gi) {
            const int s = gi % Q_STAGES, g = gi % DO_STAGES;
            // dV += P^T dO (k-step kk, queries [16kk, 16kk + 16), is warpgroup kk / 2's);
            // the item's first one overwrites dV and dK, which the previous item's
            // epilogue must have read
            if (!(ok = mbar_wait(bar(B_PR), gi & 1, ctl))) break;
            if (it == 0 && kq > 0 && !(ok = mbar_wait(bar(B_AF), (kq - 1) & 1, ctl))) break;
            tc_fence_after();
            const uint32_t dv_b = om_lo + g * STAGE_W, acc0 = it > 0 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < BT / 16; ++kk)
              umma_ts_w(tmem + DV_COL, tmem + P_COL + (kk / 2) * 16 + (kk % 2) * 8,
                        dv_b + kk * (G::KSTEP_MN >> 4), HI, idG, kk > 0 ? 1u : acc0);
            umma_commit(bar(B_PFREE));
            umma_commit(bar(B_GE(g)));
            // dK += dS^T Q
            if (!(ok = mbar_wait(bar(B_DR), gi & 1, ctl))) break;
            tc_fence_after();
            const uint32_t dk_b = qm_lo + s * STAGE_W;
#pragma unroll
            for (int kk = 0; kk < BT / 16; ++kk)
              umma_ts_w(tmem + DK_COL, tmem + DS_COL + (kk / 2) * 16 + (kk % 2) * 8,
                        dk_b + kk * (G::KSTEP_MN >> 4), HI, idG, kk > 0 ? 1u : acc0);
            umma_commit(bar(B_DSFREE));
            umma_commit(bar(B_QE(s)));
          }
          if (!ok) break;
          umma_commit(bar(B_OF));                  // this item's dV and dK are complete
        }
        ++kq;
      }
      // every MMA this thread issued has completed before TMEM is released
      umma_commit(bar(scores ? B_DONE : B_DONE2));
      mbar_wait(bar(scores ? B_DONE : B_DONE2), 0, ctl);
    }
    __syncwarp();
  } else if (warp >= 4) {
    regs_inc<kRegs64High>();                       // the compute warpgroups take what it gives back
    // ------------------------------------------------------------ compute, epilogue
    const int q = (warp - 4) >> 2;                 // query columns [32q, 32q + 32)
    const int kr = (warp & 3) * 32 + lane;         // key row (= TMEM lane)
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + S_COL + 32 * q;
    const uint32_t tP = tmem + lane_off + DP_COL + 32 * q;
    const uint32_t tPT = tmem + lane_off + P_COL + 16 * q;
    const uint32_t tDS = tmem + lane_off + DS_COL + 16 * q;
    const float2 c2 = make_float2(c_log2, c_log2);
    uint4* stage = reinterpret_cast<uint4*>(sg + SM::ST_OFF + q * 8192) + (warp & 3) * 32 * 4;
    using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    bool ok = true;
    int gi = 0, kq = 0;
    for (int k = 0; ok; ++k) {
      const int id = next_item(k, ok);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_TE(k & 1)));
      if (id < 0) break;
      const Item t = item_of(id);
      if (t.n_iter <= 0) continue;
      for (int it = 0, itl = 0; it < t.n_iter; ++it, ++gi, itl = itl + 1 == t.n_head ? 0 : itl + 1) {
        const int s = gi % Q_STAGES, g = gi % DO_STAGES;
        if (!(ok = mbar_wait_warp(bar(B_SF), gi & 1, ctl))) break;
        tc_fence_after();
        uint32_t x[32];
        tmem_ld32(tS, x);
        tmem_ld_wait_regs(x);
        tc_fence_before();
        mbar_arrive(bar(B_SFREE));                 // S^T may now receive the next tile
        if (!(ok = mbar_wait_warp(bar(B_QF(s)), (gi / Q_STAGES) & 1, ctl))) break;
        const float* Ls = reinterpret_cast<const float*>(sg + SM::L_OFF + s * 512) + 32 * q;
        // P^T = exp2(S^T c - L log2e); on the diagonal tile, zero where the query precedes
        // the key
        float p[32];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
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
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (32 * q + c < kr) p[c] = 0.f;
        }
        if (CAUSAL && window > 0 && (itl + 1) * BT - 1 >= window) {
          // window edge: zero where the query is W or more rows past the key
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (itl * BT + 32 * q + c - kr >= window) p[c] = 0.f;
        }
        // dP^T of this tile
        if (!(ok = mbar_wait_warp(bar(B_DPF), gi & 1, ctl))) break;
        tc_fence_after();
        tmem_ld32(tP, x);
        tmem_ld_wait_regs(x);
        tc_fence_before();
        mbar_arrive(bar(B_DPFREE));                // dP^T may now receive the next tile
        // P^T as 16-bit pairs, once the previous tile's dV has read its P^T
        {
          uint32_t pw[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pw[i] = pack2<BF16>(p[2 * i], p[2 * i + 1]);
          if (gi > 0 && !(ok = mbar_wait_warp(bar(B_PFREE), (gi - 1) & 1, ctl))) break;
          tc_fence_after();
          tmem_st16(tPT, pw);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(B_PR));
        // dS^T = P^T o (dP^T - D) as 16-bit pairs (D came with dO, which the dP^T MMAs
        // waited on)
        if (!(ok = mbar_wait_warp(bar(B_GF(g)), (gi / DO_STAGES) & 1, ctl))) break;
        const float* Ds = reinterpret_cast<const float*>(sg + SM::D_OFF + g * 512) + 32 * q;
        {
          uint32_t dw[16];
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4) {
            const float4 d4 = *reinterpret_cast<const float4*>(Ds + 4 * i4);
            const int c = 4 * i4;
            const float2 ds0 = mul2(make_float2(p[c], p[c + 1]),
                                    add2(make_float2(__uint_as_float(x[c]), __uint_as_float(x[c + 1])),
                                         make_float2(-d4.x, -d4.y)));
            const float2 ds1 = mul2(make_float2(p[c + 2], p[c + 3]),
                                    add2(make_float2(__uint_as_float(x[c + 2]), __uint_as_float(x[c + 3])),
                                         make_float2(-d4.z, -d4.w)));
            dw[2 * i4] = pack2<BF16>(ds0.x, ds0.y);
            dw[2 * i4 + 1] = pack2<BF16>(ds1.x, ds1.y);
          }
          // once the previous tile's dK has read its dS^T
          if (gi > 0 && !(ok = mbar_wait_warp(bar(B_DSFREE), (gi - 1) & 1, ctl))) break;
          tc_fence_after();
          tmem_st16(tDS, dw);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(B_DR));
      }
      if (!ok) break;
      // epilogue: warpgroup q stores 32 columns, dV's then dK's (scaled)
      if (!(ok = mbar_wait_warp(bar(B_OF), kq & 1, ctl))) break;
      tc_fence_after();
      constexpr int CH = HD / 32;                  // 32-column slices per tensor
      if (q < 2 * CH) {
        const int which = q / CH, col0 = 32 * (q % CH);
        const int row0 = t.kb * BT + (warp & 3) * 32;
        T* base = reinterpret_cast<T*>(which == 0 ? dV : dK) + col0;
        store_rows_staged<BF16>(
            tmem + lane_off + (which == 0 ? DV_COL : DK_COL) + col0, which == 0 ? 1.f : scale,
            stage, lane,
            [&](int r) { return base + t.sr.off(row0 + r, t.hk, Hkv, N, HD); }, t.sr.n - row0);
      }
      tc_fence_before();
      mbar_arrive(bar(B_AF));                      // dV, dK may take the next item
      ++kq;
    }
  } else {
    regs_dec<kRegs64Low>();                        // warp 3: idle
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int HD, bool BF16, bool CAUSAL>
cudaError_t launch_dkdv64_t(const BwdArgs& a, cudaStream_t st) {
  const int Np = (a.N + 127) / 128 * 128;
  const float* Lp = a.Dvec + static_cast<size_t>(a.BH) * Np;
  const long long nblk_kv = static_cast<long long>(Np / BT) * (a.BH / a.group);
  auto kern = dkdv64_kernel<HD, BF16, CAUSAL>;
  constexpr int smem = kv64::Smem<HD>::SMEM_BYTES;
  cudaError_t e = check_split_regs(reinterpret_cast<const void*>(kern), kRegs64Launch);
  if (e != cudaSuccess) return e;
  e = ensure_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  // an item streams the Q and dO tiles of its K/V head's query heads
  const int ord_g = order_group(a.BH / a.group, 2ll * Np * HD * 2 * a.group);
  trace_begin(TR_BWD_DKDV, st);
  e = launch_dependent(kern, static_cast<unsigned>(nblk_kv), THREADS, smem, st, a.tmQ, a.tmK,
                       a.tmV, a.tmdO, static_cast<const float*>(a.Dvec), Lp, a.dK, a.dV, a.N, Np,
                       a.group, a.window, a.cu_seqlens, a.H, a.total, a.scale, a.c_log2, ord_g,
                       a.ctl);
  trace_end(TR_BWD_DKDV, st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// ============================================================== dQ
namespace q64 {
// Q and dO (with the tile's L*log2e and D) of two work items; K and V in a 3-stage ring
// that runs on across items; dQ rows staged for the store.
template <int HD>
struct Smem {
  static constexpr int TILE = BT * HD * 2;
  static constexpr int KV_STAGES = 3;
  static constexpr int Q_OFF = 0;                           // Q of two items
  static constexpr int DO_OFF = 2 * TILE;                   // dO of two items
  static constexpr int LD_OFF = 4 * TILE;                   // per item: 128 L*log2e, 128 D
  static constexpr int K_OFF = LD_OFF + 2 * 1024;
  static constexpr int V_OFF = K_OFF + KV_STAGES * TILE;
  static constexpr int ST_OFF = V_OFF + KV_STAGES * TILE;   // 32-column row slices, 8 KiB
  static constexpr int BAR_OFF = ST_OFF + 4 * 8192;          // per compute warpgroup
  // qd_full[2], qd_empty[2], kv_full[3], kv_empty[3], s_full, s_free, dp_full, dp_free,
  // ds_full, z_free, out_full[2], acc_free[2], done[2], tile_full[2], tile_empty[2], clc
  static constexpr int NBARS = 4 + 2 * KV_STAGES + 6 + 4 + 2 + 4 + 1;
  static constexpr int CLC_OFF = (BAR_OFF + NBARS * 8 + 15) / 16 * 16;
  static constexpr int SLOT_OFF = CLC_OFF + 16;
  static constexpr int SMEM_BYTES = SLOT_OFF + 16;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA exceeds 227 KiB");
};
// TMEM: dQ of accumulator buffer a at columns 64a (HD of its 64 in use) | S (128) |
// dP (128) | Z (64: dS as 16-bit pairs).  Compute warpgroup q owns key columns
// [32q, 32q + 32) of S and dP and pair columns [16q, 16q + 16) of Z.
constexpr uint32_t S_COL = 128, DP_COL = 256, Z_COL = 384;

// One 128-query tile of one query head and the key blocks it sees.
struct Item {
  int bh, qb, hq, hk, j_lo, n_iter;
  SeqRows sr;
};
template <bool CAUSAL, bool WINDOW, bool PACKED>
__device__ __forceinline__ Item item(int id, int nqb, int ord_g, int N, int group, int window,
                                     const int* __restrict__ cu_seqlens, int H, int total) {
  Item t;
  const BlockPos bp = block_pos(nqb, id, ord_g);
  t.bh = bp.bh;
  t.qb = nqb - 1 - bp.rank;                       // causal: the last query tiles have the most work
  t.j_lo = WINDOW ? max(0, t.qb * BT - window + 1) / BT : 0;
  t.sr = seq_rows_t<PACKED>(cu_seqlens, t.bh / H, N, total);
  t.hq = t.sr.packed ? t.bh % H : t.bh;
  t.hk = t.sr.packed ? (t.bh % H) / group : t.bh / group;
  const int nk_r = (t.sr.n + BT - 1) / BT;        // key blocks of this sequence
  t.n_iter = t.qb * BT >= t.sr.n ? 0 : (CAUSAL ? min(t.qb + 1, nk_r) : nk_r) - t.j_lo;
  if (t.n_iter < 0) t.n_iter = 0;
  return t;
}
}  // namespace q64

template <int HD, bool BF16, bool CAUSAL, bool WINDOW, bool PACKED>
__global__ void __launch_bounds__(THREADS, 1)
    dq64_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                const float* __restrict__ Dp, const float* __restrict__ Lp, void* __restrict__ dQ,
                int N, int Np, int group, int window, const int* __restrict__ cu_seqlens, int H,
                int total, float scale, float c_log2, int ord_g, KernelCtl ctl) {
  using namespace q64;
  using SM = Smem<HD>;
  using G = Geo<HD>;
  constexpr int TILE = SM::TILE, KV_STAGES = SM::KV_STAGES;
  extern __shared__ __align__(1024) uint8_t sg[];
  const uint32_t sb = smem_u32(sg);
  grid_dep_launch();
  if (sb & 1023u) {                                // see FA_DEV_SMEM_ALIGN
    grid_dep_wait();
    if (threadIdx.x == 0) atomicOr(ctl.status, FA_DEV_SMEM_ALIGN);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = Np / BT;
  auto item_of = [&](int id) {
    return item<CAUSAL, WINDOW, PACKED>(id, nqb, ord_g, N, group, window, cu_seqlens, H, total);
  };

  auto bar = [&](int i) -> uint32_t { return sb + SM::BAR_OFF + 8 * i; };
  auto B_QDF = [&](int b) { return b; };
  auto B_QDE = [&](int b) { return 2 + b; };
  auto B_KF = [&](int s) { return 4 + s; };
  auto B_KE = [&](int s) { return 4 + KV_STAGES + s; };
  const int B_SF = 4 + 2 * KV_STAGES, B_SFREE = B_SF + 1, B_DPF = B_SF + 2, B_DPFREE = B_SF + 3,
            B_DSF = B_SF + 4, B_ZFREE = B_SF + 5;
  auto B_OF = [&](int a) { return B_SF + 6 + a; };
  auto B_AF = [&](int a) { return B_SF + 8 + a; };
  auto B_DONE = [&](int i) { return B_SF + 10 + i; };
  auto B_TF = [&](int b) { return B_SF + 12 + b; };
  auto B_TE = [&](int b) { return B_SF + 14 + b; };
  const int B_CLC = B_SF + 16;
  volatile int* slot = reinterpret_cast<volatile int*>(sg + SM::SLOT_OFF + 4);
  const uint32_t clc_resp = sb + SM::CLC_OFF;

  if (threadIdx.x == 0) {
    for (int i = 0; i < SM::NBARS; ++i) mbar_init(bar(i), 1);
    mbar_init(bar(B_SFREE), 512);
    mbar_init(bar(B_DPFREE), 512);
    mbar_init(bar(B_DSF), 512);
    mbar_init(bar(B_AF(0)), 512);
    mbar_init(bar(B_AF(1)), 512);
    for (int i = 0; i < KV_STAGES; ++i) mbar_init(bar(B_KE(i)), 2);   // both MMA issuers
    mbar_init(bar(B_QDE(0)), 1);
    mbar_init(bar(B_QDE(1)), 1);
    mbar_init(bar(B_TE(0)), 18);                   // the MMA issuers and one lane per compute warp
    mbar_init(bar(B_TE(1)), 18);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sb + SM::SLOT_OFF, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sg + SM::SLOT_OFF);
  grid_dep_wait();                                 // D and L*log2e from the pre-pass

  auto next_item = [&](int k, bool& ok) -> int {
    if (!(ok = mbar_wait(bar(B_TF(k & 1)), (k >> 1) & 1, ctl))) return -1;
    return slot[k & 1];
  };

  if (warp == 0) {
    regs_dec<kRegs64Low>();                        // warpgroup 0 (TMA, MMA issue): few registers
    // ------------------------------------------------------------ producer, scheduler
    if (lane == 0) {
      bool ok = true, pending = false;
      int id = static_cast<int>(blockIdx.x);
      int gj = 0, kq = 0, nkv = 0, n_req = 0;     // K/V tiles, items, K/V loads issued, requests
      for (int k = 0; ok; ++k) {
        if (!(ok = mbar_wait(bar(B_TE(k & 1)), ((k >> 1) & 1) ^ 1, ctl))) break;
        slot[k & 1] = id;
        mbar_arrive(bar(B_TF(k & 1)));
        if (id < 0) break;
        // ask for the next item together with this item's last loads (as in dK/dV)
        auto request = [&]() {
          mbar_arrive_expect_tx(bar(B_CLC), 16);
          clc_try_cancel(clc_resp, bar(B_CLC));
          pending = true;
          ++n_req;
        };
        const Item t = item_of(id);
        if (t.n_iter <= 0) request();
        if (t.n_iter > 0) {
          const int b = kq & 1;
          const int qrow = t.qb * BT;
          if (!(ok = mbar_wait(bar(B_QDE(b)), ((kq >> 1) & 1) ^ 1, ctl))) break;
          mbar_arrive_expect_tx(bar(B_QDF(b)), 2 * TILE + 1024);
          for (int c = 0; c < G::NCH; ++c) {
            tma_load_3d(sb + SM::Q_OFF + b * TILE + c * G::CHUNK, &tmQ, bar(B_QDF(b)),
                        c * G::SPAN, t.sr.y(qrow, t.hq), t.sr.z(qrow, t.hq));
            tma_load_3d(sb + SM::DO_OFF + b * TILE + c * G::CHUNK, &tmdO, bar(B_QDF(b)),
                        c * G::SPAN, t.sr.y(qrow, t.hq), t.sr.z(qrow, t.hq));
          }
          const size_t row = static_cast<size_t>(t.bh) * Np + qrow;
          bulk_load(sb + SM::LD_OFF + b * 1024, Lp + row, 512, bar(B_QDF(b)));
          bulk_load(sb + SM::LD_OFF + b * 1024 + 512, Dp + row, 512, bar(B_QDF(b)));
          ++kq;
          for (int j = 0; j < t.n_iter; ++j, ++gj) {
            const int s = gj % KV_STAGES;
            const int krow = (t.j_lo + j) * BT;
            if (!(ok = mbar_wait(bar(B_KE(s)), ((gj / KV_STAGES) & 1) ^ 1, ctl))) break;
            mbar_arrive_expect_tx(bar(B_KF(s)), 2 * TILE);
            for (int c = 0; c < G::NCH; ++c) {
              tma_load_3d(sb + SM::K_OFF + s * TILE + c * G::CHUNK, &tmK, bar(B_KF(s)),
                          c * G::SPAN, t.sr.y(krow, t.hk), t.sr.z(krow, t.hk));
              tma_load_3d(sb + SM::V_OFF + s * TILE + c * G::CHUNK, &tmV, bar(B_KF(s)),
                          c * G::SPAN, t.sr.y(krow, t.hk), t.sr.z(krow, t.hk));
            }
            ++nkv;
            if (j + 1 == t.n_iter) request();
          }
          if (!ok) break;
        }
        // the next item: a CTA that had not started, if any was left
        if (!(ok = mbar_wait(bar(B_CLC), k & 1, ctl))) break;
        pending = false;
        id = clc_result(clc_resp);
      }
      if (!ok) {
        // drain: wait (bounded) for the copies this thread may still have in flight
        if (pending) mbar_wait(bar(B_CLC), (n_req - 1) & 1, ctl);   // the response lands in smem
        for (int i = max(0, kq - 2); i < kq; ++i) mbar_wait(bar(B_QDF(i & 1)), (i >> 1) & 1, ctl);
        for (int i = max(0, nkv - KV_STAGES); i < nkv; ++i)
          mbar_wait(bar(B_KF(i % KV_STAGES)), (i / KV_STAGES) & 1, ctl);
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    regs_dec<kRegs64Low>();
    // ------------------------------------------------------------ MMA issuers
    // warp 1: the score products S = Q K^T and dP = dO V^T; warp 2: dQ += dS K.  A K/V
    // stage is free once both threads' products that read it have completed.
    if (lane == 0) {
      const bool scores = warp == 1;
      constexpr uint32_t idS = umma_idesc_f16(BT, BT, BF16, false, false);   // S, dP
      constexpr uint32_t idQ = umma_idesc_f16(BT, HD, BF16, false, true);    // dQ
      constexpr uint32_t HI = G::HI, STAGE_W = TILE >> 4;
      const uint32_t q_lo = sdesc_lo(sb + SM::Q_OFF, 16), o_lo = sdesc_lo(sb + SM::DO_OFF, 16);
      const uint32_t k_lo = sdesc_lo(sb + SM::K_OFF, 16), km_lo = sdesc_lo(sb + SM::K_OFF, G::CHUNK);
      const uint32_t v_lo = sdesc_lo(sb + SM::V_OFF, 16);
      bool ok = true;
      int gj = 0, kq = 0;
      for (int k = 0; ok; ++k) {
        const int id = next_item(k, ok);
        if (!ok) break;
        mbar_arrive(bar(B_TE(k & 1)));
        if (id < 0) break;
        const Item t = item_of(id);
        if (t.n_iter <= 0) continue;
        const int b = kq & 1, a = kq & 1;
        if (scores) {
          if (!(ok = mbar_wait(bar(B_QDF(b)), (kq >> 1) & 1, ctl))) break;
          const uint32_t qa = q_lo + b * STAGE_W, oa = o_lo + b * STAGE_W;
          for (int j = 0; ok && j < t.n_iter; ++j, ++gj) {
            const int s = gj % KV_STAGES;
            if (!(ok = mbar_wait(bar(B_KF(s)), (gj / KV_STAGES) & 1, ctl))) break;
            // S once the compute warps have read the previous one, then dP likewise
            if (gj > 0 && !(ok = mbar_wait(bar(B_SFREE), (gj - 1) & 1, ctl))) break;
            tc_fence_after();
            issue_ab_t_w<HD>(tmem + S_COL, qa, k_lo + s * STAGE_W, idS);
            umma_commit(bar(B_SF));
            if (gj > 0 && !(ok = mbar_wait(bar(B_DPFREE), (gj - 1) & 1, ctl))) break;
            tc_fence_after();
            issue_ab_t_w<HD>(tmem + DP_COL, oa, v_lo + s * STAGE_W, idS);
            umma_commit(bar(B_DPF));
            umma_commit(bar(B_KE(s)));
          }
          if (!ok) break;
          umma_commit(bar(B_QDE(b)));              // this item's Q and dO no longer read
        } else {
          const uint32_t dq_col = tmem + 64 * a;
          for (int j = 0; ok && j < t.n_iter; ++j, ++gj) {
            const int s = gj % KV_STAGES;
            // dQ += dS K: dS from Z (k-step kk, keys [16kk, 16kk + 16), is warpgroup kk / 2's),
            // K as an MN-major B; the item's first one overwrites this dQ buffer, whose
            // previous item the epilogue must have read
            if (!(ok = mbar_wait(bar(B_DSF), gj & 1, ctl))) break;
            if (j == 0 && !(ok = mbar_wait(bar(B_AF(a)), ((kq >> 1) & 1) ^ 1, ctl))) break;
            tc_fence_after();
            const uint32_t kb0 = km_lo + s * STAGE_W, acc0 = j > 0 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < BT / 16; ++kk)
              umma_ts_w(dq_col, tmem + Z_COL + (kk / 2) * 16 + (kk % 2) * 8,
                        kb0 + kk * (G::KSTEP_MN >> 4), HI, idQ, kk > 0 ? 1u : acc0);
            umma_commit(bar(B_ZFREE));
            umma_commit(bar(B_KE(s)));
          }
          if (!ok) break;
          umma_commit(bar(B_OF(a)));               // this item's dQ is complete
        }
        ++kq;
      }
      // every MMA this thread issued has completed before TMEM is released
      umma_commit(bar(B_DONE(scores ? 0 : 1)));
      mbar_wait(bar(B_DONE(scores ? 0 : 1)), 0, ctl);
    }
    __syncwarp();
  } else if (warp >= 4) {
    regs_inc<kRegs64High>();                       // the compute warpgroups take what it gives back
    // ------------------------------------------------------------ compute, epilogue
    const int q = (warp - 4) >> 2;                 // key columns [32q, 32q + 32)
    const int r = (warp & 3) * 32 + lane;          // query row within the tile (= TMEM lane)
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + S_COL + 32 * q;
    const uint32_t tP = tmem + lane_off + DP_COL + 32 * q;
    const uint32_t tZ = tmem + lane_off + Z_COL + 16 * q;
    uint4* stage = reinterpret_cast<uint4*>(sg + SM::ST_OFF + q * 8192) + (warp & 3) * 32 * 4;
    using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    const float2 c2 = make_float2(c_log2, c_log2);
    bool ok = true;
    int gj = 0, kq = 0;
    for (int k = 0; ok; ++k) {
      const int id = next_item(k, ok);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_TE(k & 1)));
      if (id < 0) break;
      const Item t = item_of(id);
      if (t.n_iter <= 0) continue;
      const int b = kq & 1, a = kq & 1;
      const int grow = t.qb * BT + r;
      // this row's L*log2e and D (padded rows: +inf and 0, never stored)
      if (!(ok = mbar_wait_warp(bar(B_QDF(b)), (kq >> 1) & 1, ctl))) break;
      const float lr = reinterpret_cast<const float*>(sg + SM::LD_OFF + b * 1024)[r];
      const float dr = reinterpret_cast<const float*>(sg + SM::LD_OFF + b * 1024 + 512)[r];
      const float lsub = lr == INFINITY ? 0.f : lr;
      const float2 nl2 = make_float2(-lsub, -lsub), nd2 = make_float2(-dr, -dr);
      for (int j = 0; j < t.n_iter; ++j, ++gj) {
        const int k0 = (t.j_lo + j) * BT + 32 * q;  // first key of this thread's columns
        if (!(ok = mbar_wait_warp(bar(B_SF), gj & 1, ctl))) break;
        tc_fence_after();
        uint32_t x[32];
        tmem_ld32(tS, x);
        tmem_ld_wait_regs(x);
        tc_fence_before();
        mbar_arrive(bar(B_SFREE));                 // S may now receive the next block
        // P = exp2(S c - L log2e); on the diagonal block, zero where the key follows the query
        float p[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 tt = fma2(make_float2(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1])),
                                 c2, nl2);
          p[2 * i] = ex2(tt.x);
          p[2 * i + 1] = ex2(tt.y);
        }
        if (CAUSAL && t.j_lo + j == t.qb) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (k0 + c > grow) p[c] = 0.f;
        }
        if (WINDOW && t.qb * BT + BT - 1 - (t.j_lo + j) * BT >= window) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (grow - (k0 + c) >= window) p[c] = 0.f;
        }
        if (PACKED && k0 + 32 > t.sr.n) {
          // keys past the end of a packed sequence are the next sequence's keys
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (k0 + c >= t.sr.n) p[c] = 0.f;
        }
        if (!(ok = mbar_wait_warp(bar(B_DPF), gj & 1, ctl))) break;
        tc_fence_after();
        tmem_ld32(tP, x);
        tmem_ld_wait_regs(x);
        tc_fence_before();
        mbar_arrive(bar(B_DPFREE));                // dP may now receive the next block
        // dS = P o (dP - D) as 16-bit pairs into Z once the previous block's dQ read it
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 ds = mul2(make_float2(p[2 * i], p[2 * i + 1]),
                                 add2(make_float2(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1])),
                                      nd2));
          w[i] = pack2<BF16>(ds.x, ds.y);
        }
        if (gj > 0 && !(ok = mbar_wait_warp(bar(B_ZFREE), (gj - 1) & 1, ctl))) break;
        tc_fence_after();
        tmem_st16(tZ, w);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(B_DSF));
      }
      if (!ok) break;
      // epilogue: warpgroup q stores dQ columns [32q, 32q + 32) (scaled) from buffer a
      if (!(ok = mbar_wait_warp(bar(B_OF(a)), (kq >> 1) & 1, ctl))) break;
      tc_fence_after();
      if (32 * q < HD) {
        const int row0 = t.qb * BT + (warp & 3) * 32;
        T* base = reinterpret_cast<T*>(dQ) + 32 * q;
        store_rows_staged<BF16>(
            tmem + lane_off + 64 * a + 32 * q, scale, stage, lane,
            [&](int rr) { return base + t.sr.off(row0 + rr, t.hq, H, N, HD); }, t.sr.n - row0);
      }
      tc_fence_before();
      mbar_arrive(bar(B_AF(a)));                   // buffer a may take the item after next
      ++kq;
    }
  } else {
    regs_dec<kRegs64Low>();                        // warp 3: idle
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int HD, bool BF16, bool CAUSAL>
cudaError_t launch_dq64_t(const BwdArgs& a, cudaStream_t st) {
  const int Np = (a.N + 127) / 128 * 128;
  const float* Lp = a.Dvec + static_cast<size_t>(a.BH) * Np;
  const long long nblk = static_cast<long long>(Np / BT) * a.BH;           // per query head
  // windowed and packed-sequence kernels are separate instantiations
  auto kern = CAUSAL && a.window > 0
      ? (a.cu_seqlens ? dq64_kernel<HD, BF16, CAUSAL, CAUSAL, true>
                      : dq64_kernel<HD, BF16, CAUSAL, CAUSAL, false>)
      : (a.cu_seqlens ? dq64_kernel<HD, BF16, CAUSAL, false, true>
                      : dq64_kernel<HD, BF16, CAUSAL, false, false>);
  constexpr int smem = q64::Smem<HD>::SMEM_BYTES;
  cudaError_t e = check_split_regs(reinterpret_cast<const void*>(kern), kRegs64Launch);
  if (e != cudaSuccess) return e;
  e = ensure_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  // an item streams the K and V tiles of its query head's K/V head
  const int ord_g = order_group(a.BH, 2ll * Np * HD * 2);
  trace_begin(TR_BWD_DQ, st);
  e = launch_dependent(kern, static_cast<unsigned>(nblk), THREADS, smem, st, a.tmQ, a.tmK, a.tmV,
                       a.tmdO, static_cast<const float*>(a.Dvec), Lp, a.dQ, a.N, Np, a.group,
                       a.window, a.cu_seqlens, a.H, a.total, a.scale, a.c_log2, ord_g, a.ctl);
  trace_end(TR_BWD_DQ, st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_dkdv64(const BwdArgs& a, int d, bool bf16, bool causal, cudaStream_t st) {
  if (d == 32) {
    if (bf16) return causal ? launch_dkdv64_t<32, true, true>(a, st) : launch_dkdv64_t<32, true, false>(a, st);
    return causal ? launch_dkdv64_t<32, false, true>(a, st) : launch_dkdv64_t<32, false, false>(a, st);
  }
  if (d == 64) {
    if (bf16) return causal ? launch_dkdv64_t<64, true, true>(a, st) : launch_dkdv64_t<64, true, false>(a, st);
    return causal ? launch_dkdv64_t<64, false, true>(a, st) : launch_dkdv64_t<64, false, false>(a, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_dq64(const BwdArgs& a, int d, bool bf16, bool causal, cudaStream_t st) {
  if (d == 32) {
    if (bf16) return causal ? launch_dq64_t<32, true, true>(a, st) : launch_dq64_t<32, true, false>(a, st);
    return causal ? launch_dq64_t<32, false, true>(a, st) : launch_dq64_t<32, false, false>(a, st);
  }
  if (d == 64) {
    if (bf16) return causal ? launch_dq64_t<64, true, true>(a, st) : launch_dq64_t<64, true, false>(a, st);
    return causal ? launch_dq64_t<64, false, true>(a, st) : launch_dq64_t<64, false, false>(a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fa
