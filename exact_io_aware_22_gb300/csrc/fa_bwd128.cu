// fa_bwd128.cu -- fused attention backward for head dim 128 on sm_103a.
//
// Method: "flash-attn-triton" docs page, section "Scope" (backward kernels for
// dQ, dK, dV that rebuild P from the saved L; causal mask only on diagonal
// tiles; ragged N) and "Source" (delta pre-pass, then dK/dV and dQ).  Gradients
// follow the chain rule of the forward:
//   P = exp(S - L),  dV = P^T dO,  dP = dO V^T,  D = rowsum(dO o O),
//   dS = P o (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
//
// One CTA per 128-key block (K, V stay in shared memory); the loop runs over
// 64-query tiles (causal: from the diagonal down).  Per tile, five tcgen05
// products, accumulators in TMEM (512 columns):
//   [  0,128) dV += P^T dO        A = P^T from TMEM (double-buffered), B = dO
//   [128,256) dK += dS^T Q        A = dS^T swizzled in smem (double-buffered)
//   [256,320) S^T  = K Q^T        fp32, 128 keys x 64 queries
//   [320,384) dP^T = V dO^T
//   [384,448) dQ^T = K^T dS^T     fp32, 128 (head dim) x 64 queries
//   [448,512) P^T, two buffers of 32 columns (64 packed 16-bit queries)
// Roles (512 threads, one CTA per SM):
//   warp 0       TMA producer: K, V once; Q, dO tiles plus their L, D into a ring.
//   warp 1       TMEM allocator; lane 0 issues every MMA and commit.
//   warps 4-11   two compute warpgroups, one thread per key row, 32 query
//                columns each: rebuild P^T and dS^T from S^T, dP^T, L, D.
//   warps 12-15  dQ warpgroup, one thread per head-dim row of dQ^T: takes the
//                tile out of TMEM and adds it into the fp32 dQ accumulator with
//                fp32 reductions at L2 (each warp instruction covers 32
//                consecutive head-dim floats of one query row).  Going straight
//                from registers keeps the tile out of shared memory, whose
//                bandwidth the N = 64 MMAs already saturate.
// The compute warps release S^T / dP^T as soon as they hold them in registers,
// so the next tile's S^T, dP^T MMAs overlap this tile's softmax-like work, and
// this tile's dV, dK, dQ^T MMAs overlap the next tile's.
#include "fa_internal.h"
#include "fa_ptx.cuh"

#include <type_traits>

namespace fa {

namespace {

constexpr int HD = 128;          // head dim
constexpr int BN = 128;          // keys per CTA
constexpr int BQ = 64;           // queries per iteration
constexpr int THREADS = 512;
constexpr int STAGES = 3;
constexpr float LOG2E = 1.4426950408889634f;

constexpr int KT_BYTES = BN * HD * 2;           // K or V tile: two 64-column chunks
constexpr int KT_CHUNK = BN * 128;              // 16 KiB
constexpr int QT_BYTES = BQ * HD * 2;           // Q or dO tile: two 64-column chunks
constexpr int QT_CHUNK = BQ * 128;              // 8 KiB
constexpr int DS_BYTES = BN * BQ * 2;           // dS^T tile: one 128-byte row per key
constexpr int K_OFF = 0;
constexpr int V_OFF = KT_BYTES;
constexpr int Q_OFF = 2 * KT_BYTES;
constexpr int DO_OFF = Q_OFF + STAGES * QT_BYTES;
constexpr int DS_OFF = DO_OFF + STAGES * QT_BYTES;
constexpr int LD_OFF = DS_OFF + 2 * DS_BYTES;   // per stage: 64 L*log2e, then 64 D
constexpr int BAR_OFF = LD_OFF + STAGES * 512;
// kv_full, q_full[S], q_empty[S], s_full, sp_free, p_full[2], dq_full, dq_empty, o_full, done.
// p_full alternates by tile parity: the compute warps may finish tile i+1 before the MMA
// thread has observed tile i, and one barrier would then have run two phases ahead.
constexpr int NBARS = 1 + 2 * STAGES + 8;
constexpr int SLOT_OFF = BAR_OFF + NBARS * 8;
constexpr int SMEM_BYTES = SLOT_OFF + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA exceeds 227 KiB");

constexpr uint32_t DV_COL = 0, DK_COL = 128, S_COL = 256, DP_COL = 320, DQ_COL = 384,
                   P_COL = 448;

// 1-D bulk copy global -> shared, completing on an mbarrier (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}
template <bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(THREADS, 1)
    bwd128_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  float* __restrict__ dQacc, const float* __restrict__ Dp,
                  const float* __restrict__ Lp, void* __restrict__ dK, void* __restrict__ dV,
                  int N, int Np, float scale, float c_log2, KernelCtl ctl) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* sg = smem_raw + (sb - raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = (N + BN - 1) / BN;
  const int nq = (N + BQ - 1) / BQ;
  const int bh = blockIdx.x / nkb;
  const int kb = blockIdx.x % nkb;                 // causal: block 0 has the most work, runs first
  const int q_start = CAUSAL ? kb * (BN / BQ) : 0;
  const int n_iter = nq - q_start;

  auto bar = [&](int i) -> uint32_t { return sb + BAR_OFF + 8 * i; };
  const int B_KV = 0;
  auto B_QF = [&](int s) { return 1 + s; };
  auto B_QE = [&](int s) { return 1 + STAGES + s; };
  const int B_SF = 1 + 2 * STAGES, B_SPF = B_SF + 1, B_DQF = B_SF + 2, B_DQE = B_SF + 3,
            B_OF = B_SF + 4, B_DONE = B_SF + 5;
  auto B_PF = [&](int b) { return B_SF + 6 + b; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBARS; ++i) mbar_init(bar(i), 1);
    mbar_init(bar(B_SPF), 256);
    mbar_init(bar(B_PF(0)), 256);
    mbar_init(bar(B_PF(1)), 256);
    mbar_init(bar(B_DQE), 128);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (n_iter > 0) {
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(B_KV), 2 * KT_BYTES);
        for (int c = 0; c < 2; ++c) {
          tma_load_3d(sb + K_OFF + c * KT_CHUNK, &tmK, bar(B_KV), c * 64, kb * BN, bh);
          tma_load_3d(sb + V_OFF + c * KT_CHUNK, &tmV, bar(B_KV), c * 64, kb * BN, bh);
        }
      }
      bool ok = true;
      int it = 0;
      if (lane == 0) {
        for (; it < n_iter; ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!(ok = mbar_wait(bar(B_QE(s)), ph ^ 1, ctl))) break;
          const int qrow = (q_start + it) * BQ;
          mbar_arrive_expect_tx(bar(B_QF(s)), 2 * QT_BYTES + 512);
          for (int c = 0; c < 2; ++c) {
            tma_load_3d(sb + Q_OFF + s * QT_BYTES + c * QT_CHUNK, &tmQ, bar(B_QF(s)), c * 64, qrow,
                        bh);
            tma_load_3d(sb + DO_OFF + s * QT_BYTES + c * QT_CHUNK, &tmdO, bar(B_QF(s)), c * 64,
                        qrow, bh);
          }
          // L*log2e and D of the 64 queries (padded per-row arrays, 256-byte aligned rows)
          const size_t row = static_cast<size_t>(bh) * Np + qrow;
          bulk_load(sb + LD_OFF + s * 512, Lp + row, 256, bar(B_QF(s)));
          bulk_load(sb + LD_OFF + s * 512 + 256, Dp + row, 256, bar(B_QF(s)));
        }
      }
      if (!ok && lane == 0) {
        mbar_wait(bar(B_KV), 0, ctl);
        for (int jj = max(0, it - STAGES); jj < it; ++jj)
          mbar_wait(bar(B_QF(jj % STAGES)), (jj / STAGES) & 1, ctl);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_iter > 0) {
      constexpr uint32_t idS = umma_idesc_f16(BN, BQ, BF16, false, false);   // S^T, dP^T
      constexpr uint32_t idG = umma_idesc_f16(BN, HD, BF16, false, true);    // dV, dK
      constexpr uint32_t idQ = umma_idesc_f16(HD, BQ, BF16, true, true);     // dQ^T
      auto issue_sdp = [&](int it) {
        const int s = it % STAGES;
        const uint32_t qa = sb + Q_OFF + s * QT_BYTES, da = sb + DO_OFF + s * QT_BYTES;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t ok_ = (kk / 4) * KT_CHUNK + (kk % 4) * 32;
          const uint32_t oq = (kk / 4) * QT_CHUNK + (kk % 4) * 32;
          umma_ss(tmem + S_COL, umma_sdesc(sb + K_OFF + ok_, 16, 1024, UMMA_SW128),
                  umma_sdesc(qa + oq, 16, 1024, UMMA_SW128), idS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t ok_ = (kk / 4) * KT_CHUNK + (kk % 4) * 32;
          const uint32_t oq = (kk / 4) * QT_CHUNK + (kk % 4) * 32;
          umma_ss(tmem + DP_COL, umma_sdesc(sb + V_OFF + ok_, 16, 1024, UMMA_SW128),
                  umma_sdesc(da + oq, 16, 1024, UMMA_SW128), idS, kk > 0);
        }
      };
      bool ok = mbar_wait(bar(B_KV), 0, ctl) && mbar_wait(bar(B_QF(0)), 0, ctl);
      if (ok) {
        tc_fence_after();
        issue_sdp(0);
        umma_commit(bar(B_SF));
      }
      for (int it = 0; ok && it < n_iter; ++it) {
        const int s = it % STAGES, b = it & 1;
        const uint32_t qa = sb + Q_OFF + s * QT_BYTES, da = sb + DO_OFF + s * QT_BYTES;
        const uint32_t dsa = sb + DS_OFF + b * DS_BYTES;
        if (it + 1 < n_iter) {
          // S^T, dP^T of the next tile once the compute warps hold this tile's in registers
          if (!(ok = mbar_wait(bar(B_SPF), it & 1, ctl))) break;
          if (!(ok = mbar_wait(bar(B_QF((it + 1) % STAGES)), ((it + 1) / STAGES) & 1, ctl))) break;
          tc_fence_after();
          issue_sdp(it + 1);
          umma_commit(bar(B_SF));
        }
        if (!(ok = mbar_wait(bar(B_PF(b)), (it >> 1) & 1, ctl))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)       // dV += P^T dO
          umma_ts(tmem + DV_COL, tmem + P_COL + 32 * b + 8 * kk,
                  umma_sdesc(da + kk * 2048, QT_CHUNK, 1024, UMMA_SW128), idG,
                  (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)       // dK += dS^T Q
          umma_ss(tmem + DK_COL, umma_sdesc(dsa + kk * 32, 16, 1024, UMMA_SW128),
                  umma_sdesc(qa + kk * 2048, QT_CHUNK, 1024, UMMA_SW128), idG,
                  (it > 0 || kk > 0) ? 1u : 0u);
        if (it > 0 && !(ok = mbar_wait(bar(B_DQE), (it - 1) & 1, ctl))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)       // dQ^T = K^T dS^T
          umma_ss(tmem + DQ_COL, umma_sdesc(sb + K_OFF + kk * 2048, KT_CHUNK, 1024, UMMA_SW128),
                  umma_sdesc(dsa + kk * 2048, KT_CHUNK, 1024, UMMA_SW128), idQ, kk > 0);
        umma_commit(bar(B_DQF));
        umma_commit(bar(B_QE(s)));
      }
      if (ok) umma_commit(bar(B_OF));
      umma_commit(bar(B_DONE));
      mbar_wait(bar(B_DONE), 0, ctl);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ compute
    const int h = (warp - 4) >> 2;                 // query columns [32h, 32h + 32)
    const int kr = (warp & 3) * 32 + lane;         // key row (= TMEM lane)
    const int gkey = kb * BN + kr;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    bool ok = n_iter > 0;
    for (int it = 0; ok && it < n_iter; ++it) {
      const int s = it % STAGES, b = it & 1;
      const int q0 = (q_start + it) * BQ + 32 * h;  // first query of this thread's columns
      if (!(ok = mbar_wait(bar(B_SF), it & 1, ctl))) break;
      tc_fence_after();
      uint32_t sr[32], dp[32];
      tmem_ld32(tmem + lane_off + S_COL + 32 * h, sr);
      tmem_ld32(tmem + lane_off + DP_COL + 32 * h, dp);
      tmem_ld_wait_regs(sr);
      tmem_ld_wait_regs(dp);
      tc_fence_before();
      mbar_arrive(bar(B_SPF));
      if (!(ok = mbar_wait(bar(B_QF(s)), (it / STAGES) & 1, ctl))) break;
      const float4* L4 = reinterpret_cast<const float4*>(sg + LD_OFF + s * 512 + 32 * h * 4);
      const float4* D4 = reinterpret_cast<const float4*>(sg + LD_OFF + s * 512 + 256 + 32 * h * 4);
      const bool diag = CAUSAL && it < BN / BQ;
      uint32_t pw[16];
      uint8_t* ds_row = sg + DS_OFF + b * DS_BYTES + kr * 128;
#pragma unroll
      for (int u = 0; u < 4; ++u) {                // 8 queries = one 16-byte chunk of dS^T
        const float4 la = L4[2 * u], lb = L4[2 * u + 1];
        const float4 da = D4[2 * u], db = D4[2 * u + 1];
        const float lq[8] = {la.x, la.y, la.z, la.w, lb.x, lb.y, lb.z, lb.w};
        const float dq[8] = {da.x, da.y, da.z, da.w, db.x, db.y, db.z, db.w};
        float p[8], ds[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int c = 8 * u + e;
          float pv = ex2(fmaf(__uint_as_float(sr[c]), c_log2, -lq[e]));
          if (diag && q0 + c < gkey) pv = 0.f;
          p[e] = pv;
          ds[e] = pv * (__uint_as_float(dp[c]) - dq[e]);
        }
        uint32_t dw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          pw[4 * u + e] = pack2<BF16>(p[2 * e], p[2 * e + 1]);
          dw[e] = pack2<BF16>(ds[2 * e], ds[2 * e + 1]);
        }
        const int chunk = 4 * h + u;               // 128-byte swizzle: chunk ^ (row & 7)
        *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (kr & 7)) << 4)) =
            make_uint4(dw[0], dw[1], dw[2], dw[3]);
      }
      tmem_st16(tmem + lane_off + P_COL + 32 * b + 16 * h, pw);
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(B_PF(b)));
    }
    if (ok && mbar_wait(bar(B_OF), 0, ctl)) {
      tc_fence_after();
      using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
      const bool valid = gkey < N;
      const size_t roff = (static_cast<size_t>(bh) * N + gkey) * HD + 64 * h;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = (which == 0 ? DV_COL : DK_COL) + 64 * h;
        const float mul = which == 0 ? 1.f : scale;
        T* dst = reinterpret_cast<T*>(which == 0 ? dV : dK) + roff;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t v[16];
          tmem_ld16(tmem + lane_off + col + 16 * cc, v);
          tmem_ld_wait_regs(v);
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            w[i] = pack2<BF16>(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
          if (valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + 16 * cc);
            d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
            d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
          }
        }
      }
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ dQ accumulation
    const int dr = (warp & 3) * 32 + lane;         // head-dim row of dQ^T (= TMEM lane)
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    float* acc = dQacc + static_cast<size_t>(bh) * Np * HD + dr;
    bool ok = n_iter > 0;
    for (int it = 0; ok && it < n_iter; ++it) {
      if (!(ok = mbar_wait(bar(B_DQF), it & 1, ctl))) break;
      tc_fence_after();
      uint32_t v0[32], v1[32];
      tmem_ld32(tmem + lane_off + DQ_COL, v0);
      tmem_ld32(tmem + lane_off + DQ_COL + 32, v1);
      tmem_ld_wait_regs(v0);
      tmem_ld_wait_regs(v1);
      tc_fence_before();
      mbar_arrive(bar(B_DQE));
      float* row = acc + static_cast<size_t>((q_start + it) * BQ) * HD;
#pragma unroll
      for (int c = 0; c < 32; ++c) atomicAdd(row + c * HD, __uint_as_float(v0[c]));
#pragma unroll
      for (int c = 0; c < 32; ++c) atomicAdd(row + (32 + c) * HD, __uint_as_float(v1[c]));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// dQ = scale * dQacc, rounded to the 16-bit type (rows < N only).
template <bool BF16>
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ acc,
                                                         void* __restrict__ dQ, int N, int Np,
                                                         long long n8, float scale) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const long long row = i / (HD / 8);
  const int part = static_cast<int>(i % (HD / 8));
  const long long bh = row / N;
  const int r = static_cast<int>(row % N);
  const float4* src = reinterpret_cast<const float4*>(acc + ((bh * Np + r) * HD + part * 8));
  const float4 a = src[0], b = src[1];
  uint4 w;
  w.x = pack2<BF16>(a.x * scale, a.y * scale);
  w.y = pack2<BF16>(a.z * scale, a.w * scale);
  w.z = pack2<BF16>(b.x * scale, b.y * scale);
  w.w = pack2<BF16>(b.z * scale, b.w * scale);
  reinterpret_cast<uint4*>(dQ)[i] = w;
}

template <bool BF16, bool CAUSAL>
cudaError_t launch_t(const BwdArgs& a, cudaStream_t st) {
  const int Np = (a.N + 127) / 128 * 128;
  const float* Lp = a.Dvec + static_cast<size_t>(a.BH) * Np;
  auto kern = bwd128_kernel<BF16, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int nkb = (a.N + BN - 1) / BN;
  const long long grid = static_cast<long long>(nkb) * a.BH;
  trace_begin(TR_BWD_FUSED, st);
  kern<<<static_cast<unsigned>(grid), THREADS, SMEM_BYTES, st>>>(
      a.tmQ64, a.tmK, a.tmV, a.tmdO64, a.dQacc, a.Dvec, Lp, a.dK, a.dV, a.N, Np, a.scale,
      a.c_log2, a.ctl);
  trace_end(TR_BWD_FUSED, st);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long n8 = static_cast<long long>(a.BH) * a.N * (HD / 8);
  trace_begin(TR_BWD_DQCVT, st);
  dq_convert_kernel<BF16><<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, st>>>(
      a.dQacc, a.dQ, a.N, Np, n8, a.scale);
  trace_end(TR_BWD_DQCVT, st);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd128_fused(const BwdArgs& a, bool bf16, bool causal, cudaStream_t st) {
  if (bf16) return causal ? launch_t<true, true>(a, st) : launch_t<true, false>(a, st);
  return causal ? launch_t<false, true>(a, st) : launch_t<false, false>(a, st);
}

}  // namespace fa
