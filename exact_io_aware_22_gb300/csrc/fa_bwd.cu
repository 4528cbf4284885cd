// fa_bwd.cu -- exact attention backward for sm_103a.
//
// Method: "flash-attn-triton" docs page, section "Scope" (backward kernels for
// dQ, dK, dV that rebuild P from the saved L instead of storing it; causal mask
// only on diagonal tiles; ragged N) and "Source" (a delta pre-pass, then dK/dV,
// then dQ); the FlashAttention note, "Key Mechanisms" (backward recomputation).
// The pages print no gradient formulas; the chain rule of the forward gives
//   P = exp(S - L),  dV = P^T dO,  dP = dO V^T,  D = rowsum(dO o O),
//   dS = P o (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
//
// Three kernels, all on one stream (at d = 64 and 128 the pre-pass is followed by
// the kernels of fa_bwd128.cu instead of the two below, which serve d = 32):
//   pre_kernel   D = rowsum(dO o O) and L * log2(e), both laid out per 128-row
//                query block and padded (L -> +inf, D -> 0 past N) so the
//                other kernels read them with aligned vector loads.
//   dkdv_kernel  one CTA per 128-key block; K and V stay in shared memory; the
//                loop runs over query blocks (causal: from the diagonal down).
//                S^T = K Q^T and dP^T = V dO^T land in TMEM; a thread per key
//                row (two warpgroups split the 128 query columns) rebuilds
//                P^T = exp2(S^T c - L log2e) and dS^T = P^T o (dP^T - D),
//                writes P^T back over S^T in TMEM (A operand of dV += P^T dO)
//                and dS^T to shared memory (A operand of dK += dS^T Q).
//   dq_kernel    one CTA per 128-row query block; Q and dO stay in shared
//                memory; the loop runs over key blocks (causal: up to the
//                diagonal).  S and dP in TMEM, a thread per query row rebuilds
//                dS and writes it over S in TMEM, dQ += dS K accumulates in TMEM.
#include "fa_internal.h"
#include "fa_ptx.cuh"

#include <type_traits>

namespace fa {

namespace {

constexpr int BM = 128;   // query rows per block
constexpr int BN = 128;   // keys per block
constexpr int THREADS = 384;
constexpr float LOG2E = 1.4426950408889634f;

template <int D>
struct Geo {
  static constexpr int SW = D == 32 ? 64 : 128;
  static constexpr int ATOM = SW / 2;
  static constexpr int NCHUNK = D / ATOM;
  static constexpr int CHUNK_BYTES = 128 * SW;
  static constexpr int TILE_BYTES = 128 * D * 2;
  static constexpr uint32_t SWZ = D == 32 ? UMMA_SW64 : UMMA_SW128;
  static constexpr int STAGES = 2;
};

template <int D>
__device__ __forceinline__ uint32_t kmajor_koff(int kk) {
  using G = Geo<D>;
  const int e = kk * 16;
  return (e / G::ATOM) * G::CHUNK_BYTES + (e % G::ATOM) * 2;
}

template <int D>
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                          int row, int bh) {
  using G = Geo<D>;
#pragma unroll
  for (int c = 0; c < G::NCHUNK; ++c)
    tma_load_3d(dst + c * G::CHUNK_BYTES, map, bar, c * G::ATOM, row, bh);
}

// ---------------------------------------------------------------- pre-pass
// Dp[bh][r] = sum_c dO[r][c] O[r][c] (fp32), Lp[bh][r] = L[r] * log2(e), for every
// flat head bh and padded row r; rows past the end of the sequence (N, or the packed
// sequence's own length) get Dp = 0, Lp = +inf, which makes their P exactly 0.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) pre_kernel(const void* __restrict__ O,
                                                  const void* __restrict__ dO,
                                                  const float* __restrict__ L,
                                                  float* __restrict__ Dp, float* __restrict__ Lp,
                                                  int N, int Np, long long rows_p,
                                                  const int* __restrict__ cu_seqlens, int H,
                                                  int total) {
  constexpr int TPR = D / 8;   // threads per row, 16 bytes each
  const long long gt = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long rp = gt / TPR;
  const int part = static_cast<int>(gt % TPR);
  float acc = 0.f;
  long long src = -1, lsrc = -1;              // row of O / dO (in rows of D), index of L
  if (rp < rows_p) {
    const long long bh = rp / Np;
    const int r = static_cast<int>(rp % Np);
    if (cu_seqlens) {
      const int hl = static_cast<int>(bh % H);
      const SeqRows sr = seq_rows(cu_seqlens, static_cast<int>(bh / H), N, total);
      if (r < sr.n) {
        src = static_cast<long long>(sr.base + r) * H + hl;
        lsrc = static_cast<long long>(hl) * total + sr.base + r;
      }
    } else if (r < N) {
      src = lsrc = bh * N + r;
    }
  }
  if (src >= 0) {
    const uint4 a = reinterpret_cast<const uint4*>(O)[src * TPR + part];
    const uint4 b = reinterpret_cast<const uint4*>(dO)[src * TPR + part];
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = unpack2<BF16>(aw[i]), y = unpack2<BF16>(bw[i]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (rp < rows_p && part == 0) {
    Dp[rp] = src >= 0 ? acc : 0.f;
    Lp[rp] = src >= 0 ? L[lsrc] * LOG2E : INFINITY;
  }
}

// ---------------------------------------------------------------- dK / dV
template <int D>
struct DkdvCfg {
  using G = Geo<D>;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = G::TILE_BYTES;
  static constexpr int Q_OFF = 2 * G::TILE_BYTES;
  static constexpr int DO_OFF = Q_OFF + G::STAGES * G::TILE_BYTES;
  static constexpr int DS_OFF = DO_OFF + G::STAGES * G::TILE_BYTES;   // 128 x 128 16-bit, SW128
  static constexpr int BAR_OFF = DS_OFF + 128 * 128 * 2;
  // kv_full, q_full[S], q_empty[S], s_full, p_full, o_full, done
  static constexpr int NBARS = 1 + 2 * G::STAGES + 4;
  static constexpr int SLOT_OFF = BAR_OFF + NBARS * 8;
  static constexpr int SMEM_BYTES = SLOT_OFF + 16 + 1024;
  static constexpr int DV_COL = 0, DK_COL = D, S_COL = 2 * D, DP_COL = 2 * D + 128;
};

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(THREADS, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                const float* __restrict__ Dp, const float* __restrict__ Lp, void* __restrict__ dK,
                void* __restrict__ dV, int N, int Np, int group, int window,
                const int* __restrict__ cu_seqlens, int H, int total, float scale, float c_log2,
                KernelCtl ctl) {
  using G = Geo<D>;
  using C = DkdvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* sg = smem_raw + (sb - raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = (N + BN - 1) / BN;
  const BlockPos bp = block_pos(nkb);
  const int bkv = bp.bh;                    // K/V head; its query heads are bkv*group + g
  const int kb = bp.rank;                   // key block (causal: block 0 has the most work)
  const int i0 = CAUSAL ? kb : 0;           // BM == BN: the diagonal query block
  const int Hkv = H / group;
  const SeqRows sr = seq_rows(cu_seqlens, bkv / Hkv, N, total);
  const int hk = sr.packed ? bkv % Hkv : bkv;            // K/V head coordinate
  const int nq_r = (sr.n + BM - 1) / BM;                 // query blocks of this sequence
  // query blocks per query head: from the diagonal to the last one that sees a key of
  // this block (a window of W keys reaches query rows up to the block's last key + W - 1)
  const int n_head = kb * BN >= sr.n ? 0
      : ((CAUSAL && window > 0) ? min(nq_r, (kb * BN + BN - 1 + window - 1) / BM + 1) : nq_r) - i0;
  const int n_iter = group * n_head;        // every query head of the group in turn
  if (n_iter <= 0) return;                  // a key block past the end of its packed sequence

  auto bar = [&](int i) -> uint32_t { return sb + C::BAR_OFF + 8 * i; };
  const int B_KV = 0;
  auto B_QF = [&](int s) { return 1 + s; };
  auto B_QE = [&](int s) { return 1 + G::STAGES + s; };
  const int B_SF = 1 + 2 * G::STAGES, B_PF = B_SF + 1, B_OF = B_SF + 2, B_DONE = B_SF + 3;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBARS; ++i) mbar_init(bar(i), 1);
    mbar_init(bar(B_PF), 256);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sb + C::SLOT_OFF, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sg + C::SLOT_OFF);

  if (warp == 0) {
    if (lane == 0 && n_iter > 0) {
      bool ok = true;
      mbar_arrive_expect_tx(bar(B_KV), 2 * G::TILE_BYTES);
      load_tile<D>(sb + C::K_OFF, &tmK, bar(B_KV), sr.y(kb * BN, hk), sr.z(kb * BN, hk));
      load_tile<D>(sb + C::V_OFF, &tmV, bar(B_KV), sr.y(kb * BN, hk), sr.z(kb * BN, hk));
      int it = 0;
      for (; it < n_iter; ++it) {
        const int s = it % G::STAGES;
        const uint32_t ph = (it / G::STAGES) & 1;
        if (!(ok = mbar_wait(bar(B_QE(s)), ph ^ 1, ctl))) break;
        mbar_arrive_expect_tx(bar(B_QF(s)), 2 * G::TILE_BYTES);
        const int g = it / n_head;
        const int qrow = (i0 + it - g * n_head) * BM, bhq = bkv * group + g;
        const int hq = sr.packed ? bhq % H : bhq;
        load_tile<D>(sb + C::Q_OFF + s * G::TILE_BYTES, &tmQ, bar(B_QF(s)), sr.y(qrow, hq),
                     sr.z(qrow, hq));
        load_tile<D>(sb + C::DO_OFF + s * G::TILE_BYTES, &tmdO, bar(B_QF(s)), sr.y(qrow, hq),
                     sr.z(qrow, hq));
      }
      if (!ok) {
        mbar_wait(bar(B_KV), 0, ctl);
        for (int jj = max(0, it - G::STAGES); jj < it; ++jj)
          mbar_wait(bar(B_QF(jj % G::STAGES)), (jj / G::STAGES) & 1, ctl);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && n_iter > 0) {
      constexpr uint32_t idS = umma_idesc_f16(BN, BM, BF16, false, false);   // M = keys
      constexpr uint32_t idG = umma_idesc_f16(BN, D, BF16, false, true);     // dV, dK
      bool ok = mbar_wait(bar(B_KV), 0, ctl);
      for (int it = 0; ok && it < n_iter; ++it) {
        const int s = it % G::STAGES;
        if (!(ok = mbar_wait(bar(B_QF(s)), (it / G::STAGES) & 1, ctl))) break;
        tc_fence_after();
        const uint32_t qa = sb + C::Q_OFF + s * G::TILE_BYTES;
        const uint32_t da = sb + C::DO_OFF + s * G::TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = kmajor_koff<D>(kk);
          umma_ss(tmem + C::S_COL, umma_sdesc(sb + C::K_OFF + o, 16, 8 * G::SW, G::SWZ),
                  umma_sdesc(qa + o, 16, 8 * G::SW, G::SWZ), idS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = kmajor_koff<D>(kk);
          umma_ss(tmem + C::DP_COL, umma_sdesc(sb + C::V_OFF + o, 16, 8 * G::SW, G::SWZ),
                  umma_sdesc(da + o, 16, 8 * G::SW, G::SWZ), idS, kk > 0);
        }
        umma_commit(bar(B_SF));
        if (!(ok = mbar_wait(bar(B_PF), it & 1, ctl))) break;
        tc_fence_after();
        // dV += P^T dO  (P^T in TMEM, packed over S^T; dO as MN-major B)
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk) {
          const uint32_t acol = C::S_COL + (kk / 4) * 64 + (kk % 4) * 8;
          umma_ts(tmem + C::DV_COL, tmem + acol,
                  umma_sdesc(da + kk * 16 * G::SW, G::CHUNK_BYTES, 8 * G::SW, G::SWZ), idG,
                  (it > 0 || kk > 0) ? 1u : 0u);
        }
        // dK += dS^T Q  (dS^T K-major SW128 in shared memory; Q as MN-major B)
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk) {
          const uint32_t aoff = (kk / 4) * (128 * 128) + (kk % 4) * 32;
          umma_ss(tmem + C::DK_COL, umma_sdesc(sb + C::DS_OFF + aoff, 16, 1024, UMMA_SW128),
                  umma_sdesc(qa + kk * 16 * G::SW, G::CHUNK_BYTES, 8 * G::SW, G::SWZ), idG,
                  (it > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar(B_QE(s)));
      }
      if (ok) umma_commit(bar(B_OF));
      umma_commit(bar(B_DONE));
      mbar_wait(bar(B_DONE), 0, ctl);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int h = (warp - 4) >> 2;                       // query-column half
    const int kr = (warp & 3) * 32 + lane;               // key row in the block (= TMEM lane)
    const int gkey = kb * BN + kr;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::S_COL + h * 64;
    const uint32_t tP = tmem + lane_off + C::DP_COL + h * 64;
    uint8_t* ds_row = sg + C::DS_OFF + h * (128 * 128) + kr * 128;
    bool ok = n_iter > 0;
    for (int it = 0; ok && it < n_iter; ++it) {
      const int g = it / n_head;
      const int qb = i0 + it - g * n_head;
      const float* Lb = Lp + static_cast<size_t>(bkv * group + g) * Np;
      const float* Db = Dp + static_cast<size_t>(bkv * group + g) * Np;
      if (!(ok = mbar_wait_warp(bar(B_SF), it & 1, ctl))) break;
      tc_fence_after();
      uint32_t s[64], dp[64];
      tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
      tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
      tmem_ld32(tP, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
      tmem_ld32(tP + 32, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
      tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&s[0]));
      tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&s[32]));
      tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
      tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
      const int q0 = qb * BM + h * 64;                    // first query of this half
      const float4* L4 = reinterpret_cast<const float4*>(Lb + q0);
      const float4* D4 = reinterpret_cast<const float4*>(Db + q0);
      const bool diag = CAUSAL && qb == kb;
      // window edge: zero where the query is W or more rows past the key
      const bool wedge = CAUSAL && window > 0 && qb * BM + BM - 1 - kb * BN >= window;
#pragma unroll
      for (int u = 0; u < 8; ++u) {                       // 8 queries (16 bytes of dS^T) per step
        const float4 la = __ldg(L4 + 2 * u), lb = __ldg(L4 + 2 * u + 1);
        const float4 da = __ldg(D4 + 2 * u), db = __ldg(D4 + 2 * u + 1);
        const float lq[8] = {la.x, la.y, la.z, la.w, lb.x, lb.y, lb.z, lb.w};
        const float dq[8] = {da.x, da.y, da.z, da.w, db.x, db.y, db.z, db.w};
        float p[8], ds[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int c = 8 * u + e;
          float pv = ex2(fmaf(__uint_as_float(s[c]), c_log2, -lq[e]));
          if (diag && q0 + c < gkey) pv = 0.f;
          if (wedge && q0 + c - gkey >= window) pv = 0.f;
          p[e] = pv;
          ds[e] = pv * (__uint_as_float(dp[c]) - dq[e]);
        }
        uint32_t pw[4], dw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          pw[e] = pack2<BF16>(p[2 * e], p[2 * e + 1]);
          dw[e] = pack2<BF16>(ds[2 * e], ds[2 * e + 1]);
        }
        // P^T packed over this half's first 32 S^T columns
        s[4 * u + 0] = pw[0];
        s[4 * u + 1] = pw[1];
        s[4 * u + 2] = pw[2];
        s[4 * u + 3] = pw[3];
        // dS^T, 128-byte swizzle: 16-byte chunk u of row kr goes to chunk u ^ (kr & 7)
        *reinterpret_cast<uint4*>(ds_row + ((u ^ (kr & 7)) << 4)) =
            make_uint4(dw[0], dw[1], dw[2], dw[3]);
      }
      tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(B_PF));
    }
    if (ok && mbar_wait_warp(bar(B_OF), 0, ctl)) {
      tc_fence_after();
      using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
      const bool valid = gkey < sr.n;
      const size_t roff = sr.off(gkey, hk, Hkv, N, D);
      constexpr int HALF = D / 2;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = (which == 0 ? C::DV_COL : C::DK_COL) + h * HALF;
        const float mul = which == 0 ? 1.f : scale;
        T* dst = reinterpret_cast<T*>(which == 0 ? dV : dK) + roff + h * HALF;
#pragma unroll
        for (int cc = 0; cc < HALF / 16; ++cc) {
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
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- dQ
template <int D>
struct DqCfg {
  using G = Geo<D>;
  static constexpr int Q_OFF = 0;
  static constexpr int DO_OFF = G::TILE_BYTES;
  static constexpr int K_OFF = 2 * G::TILE_BYTES;
  static constexpr int V_OFF = K_OFF + G::STAGES * G::TILE_BYTES;
  static constexpr int BAR_OFF = V_OFF + G::STAGES * G::TILE_BYTES;
  // q_full, kv_full[S], kv_empty[S], s_full, ds_full, o_full, done
  static constexpr int NBARS = 1 + 2 * G::STAGES + 4;
  static constexpr int SLOT_OFF = BAR_OFF + NBARS * 8;
  static constexpr int SMEM_BYTES = SLOT_OFF + 16 + 1024;
  static constexpr int S_COL = 0, DP_COL = 128, DQ_COL = 256;
};

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(THREADS, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
              const float* __restrict__ Dp, const float* __restrict__ Lp, void* __restrict__ dQ,
              int N, int Np, int group, int window, const int* __restrict__ cu_seqlens, int H,
              int total, float scale, float c_log2, KernelCtl ctl) {
  using G = Geo<D>;
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* sg = smem_raw + (sb - raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = Np / BM;
  const BlockPos bp = block_pos(nqb);
  const int bh = bp.bh;
  const int qb = nqb - 1 - bp.rank;                // causal: the last query blocks have the most work
  // key blocks j_lo .. diagonal (a window of W keys starts at the block holding the
  // block's first row - W + 1); loop position it is key block j_lo + it
  const SeqRows sr = seq_rows(cu_seqlens, bh / H, N, total);
  const int hq = sr.packed ? bh % H : bh, hk = sr.packed ? (bh % H) / group : bh / group;
  const int nk_r = (sr.n + BN - 1) / BN;                 // key blocks of this sequence
  const int j_lo = (CAUSAL && window > 0) ? max(0, qb * BM - window + 1) / BN : 0;
  const int n_iter = qb * BM >= sr.n ? 0 : (CAUSAL ? min(qb + 1, nk_r) : nk_r) - j_lo;
  if (n_iter <= 0) return;                  // a query block past the end of its packed sequence

  auto bar = [&](int i) -> uint32_t { return sb + C::BAR_OFF + 8 * i; };
  const int B_QF = 0;
  auto B_KF = [&](int s) { return 1 + s; };
  auto B_KE = [&](int s) { return 1 + G::STAGES + s; };
  const int B_SF = 1 + 2 * G::STAGES, B_PF = B_SF + 1, B_OF = B_SF + 2, B_DONE = B_SF + 3;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBARS; ++i) mbar_init(bar(i), 1);
    mbar_init(bar(B_PF), 256);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sb + C::SLOT_OFF, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sg + C::SLOT_OFF);

  if (warp == 0) {
    if (lane == 0 && n_iter > 0) {
      bool ok = true;
      mbar_arrive_expect_tx(bar(B_QF), 2 * G::TILE_BYTES);
      load_tile<D>(sb + C::Q_OFF, &tmQ, bar(B_QF), sr.y(qb * BM, hq), sr.z(qb * BM, hq));
      load_tile<D>(sb + C::DO_OFF, &tmdO, bar(B_QF), sr.y(qb * BM, hq), sr.z(qb * BM, hq));
      int it = 0;
      for (; it < n_iter; ++it) {
        const int s = it % G::STAGES;
        const uint32_t ph = (it / G::STAGES) & 1;
        if (!(ok = mbar_wait(bar(B_KE(s)), ph ^ 1, ctl))) break;
        mbar_arrive_expect_tx(bar(B_KF(s)), 2 * G::TILE_BYTES);
        const int krow = (j_lo + it) * BN;
        load_tile<D>(sb + C::K_OFF + s * G::TILE_BYTES, &tmK, bar(B_KF(s)), sr.y(krow, hk),
                     sr.z(krow, hk));
        load_tile<D>(sb + C::V_OFF + s * G::TILE_BYTES, &tmV, bar(B_KF(s)), sr.y(krow, hk),
                     sr.z(krow, hk));
      }
      if (!ok) {
        mbar_wait(bar(B_QF), 0, ctl);
        for (int jj = max(0, it - G::STAGES); jj < it; ++jj)
          mbar_wait(bar(B_KF(jj % G::STAGES)), (jj / G::STAGES) & 1, ctl);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && n_iter > 0) {
      constexpr uint32_t idS = umma_idesc_f16(BM, BN, BF16, false, false);
      constexpr uint32_t idQ = umma_idesc_f16(BM, D, BF16, false, true);
      bool ok = mbar_wait(bar(B_QF), 0, ctl);
      for (int it = 0; ok && it < n_iter; ++it) {
        const int s = it % G::STAGES;
        if (!(ok = mbar_wait(bar(B_KF(s)), (it / G::STAGES) & 1, ctl))) break;
        tc_fence_after();
        const uint32_t ka = sb + C::K_OFF + s * G::TILE_BYTES;
        const uint32_t va = sb + C::V_OFF + s * G::TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = kmajor_koff<D>(kk);
          umma_ss(tmem + C::S_COL, umma_sdesc(sb + C::Q_OFF + o, 16, 8 * G::SW, G::SWZ),
                  umma_sdesc(ka + o, 16, 8 * G::SW, G::SWZ), idS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = kmajor_koff<D>(kk);
          umma_ss(tmem + C::DP_COL, umma_sdesc(sb + C::DO_OFF + o, 16, 8 * G::SW, G::SWZ),
                  umma_sdesc(va + o, 16, 8 * G::SW, G::SWZ), idS, kk > 0);
        }
        umma_commit(bar(B_SF));
        if (!(ok = mbar_wait(bar(B_PF), it & 1, ctl))) break;
        tc_fence_after();
        // dQ += dS K  (dS in TMEM packed over S; K as MN-major B)
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint32_t acol = C::S_COL + (kk / 4) * 64 + (kk % 4) * 8;
          umma_ts(tmem + C::DQ_COL, tmem + acol,
                  umma_sdesc(ka + kk * 16 * G::SW, G::CHUNK_BYTES, 8 * G::SW, G::SWZ), idQ,
                  (it > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar(B_KE(s)));
      }
      if (ok) umma_commit(bar(B_OF));
      umma_commit(bar(B_DONE));
      mbar_wait(bar(B_DONE), 0, ctl);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int h = (warp - 4) >> 2;                       // key-column half
    const int r = (warp & 3) * 32 + lane;                // query row in the block (= TMEM lane)
    const int grow = qb * BM + r;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::S_COL + h * 64;
    const uint32_t tP = tmem + lane_off + C::DP_COL + h * 64;
    const float lr = Lp[static_cast<size_t>(bh) * Np + grow];
    const float dr = Dp[static_cast<size_t>(bh) * Np + grow];
    // padded rows (lr = +inf) would give 0 * inf; they are never stored, keep them finite
    const float lsub = lr == INFINITY ? 0.f : lr;
    bool ok = n_iter > 0;
    for (int it = 0; ok && it < n_iter; ++it) {
      if (!(ok = mbar_wait_warp(bar(B_SF), it & 1, ctl))) break;
      tc_fence_after();
      uint32_t s[64], dp[64];
      tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
      tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
      tmem_ld32(tP, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
      tmem_ld32(tP + 32, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
      tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&s[0]));
      tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&s[32]));
      tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
      tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
      const int k0 = (j_lo + it) * BN + h * 64;
      const bool diag = CAUSAL && j_lo + it == qb;
      const bool wedge = CAUSAL && window > 0 && qb * BM + BM - 1 - (j_lo + it) * BN >= window;
      // keys past the end of the sequence: zero-filled rows when dense, but the next
      // sequence's keys when packed
      const bool kedge = k0 + 64 > sr.n;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float p0 = ex2(fmaf(__uint_as_float(s[2 * i]), c_log2, -lsub));
        float p1 = ex2(fmaf(__uint_as_float(s[2 * i + 1]), c_log2, -lsub));
        if (diag) {
          if (k0 + 2 * i > grow) p0 = 0.f;
          if (k0 + 2 * i + 1 > grow) p1 = 0.f;
        }
        if (wedge) {
          if (grow - (k0 + 2 * i) >= window) p0 = 0.f;
          if (grow - (k0 + 2 * i + 1) >= window) p1 = 0.f;
        }
        if (kedge) {
          if (k0 + 2 * i >= sr.n) p0 = 0.f;
          if (k0 + 2 * i + 1 >= sr.n) p1 = 0.f;
        }
        const float ds0 = p0 * (__uint_as_float(dp[2 * i]) - dr);
        const float ds1 = p1 * (__uint_as_float(dp[2 * i + 1]) - dr);
        s[i] = pack2<BF16>(ds0, ds1);
      }
      tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(B_PF));
    }
    if (ok && mbar_wait_warp(bar(B_OF), 0, ctl)) {
      tc_fence_after();
      using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
      constexpr int HALF = D / 2;
      T* dst = reinterpret_cast<T*>(dQ) + sr.off(grow, hq, H, N, D) + h * HALF;
#pragma unroll
      for (int cc = 0; cc < HALF / 16; ++cc) {
        uint32_t v[16];
        tmem_ld16(tmem + lane_off + C::DQ_COL + h * HALF + 16 * cc, v);
        tmem_ld_wait_regs(v);
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          w[i] = pack2<BF16>(__uint_as_float(v[2 * i]) * scale, __uint_as_float(v[2 * i + 1]) * scale);
        if (grow < sr.n) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + 16 * cc);
          d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
          d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool BF16, bool CAUSAL>
cudaError_t launch_bwd_t(const BwdArgs& a, cudaStream_t st) {
  const int nqb = (a.N + BM - 1) / BM;
  const int Np = nqb * BM;
  float* Lp = a.Dvec + static_cast<size_t>(a.BH) * Np;
  {
    const long long rows_p = static_cast<long long>(a.BH) * Np;
    const long long threads = rows_p * (D / 8);
    const long long blocks = (threads + 255) / 256;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    trace_begin(TR_BWD_PRE, st);
    pre_kernel<D, BF16><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        a.O, a.dO, a.L, a.Dvec, Lp, a.N, Np, rows_p, a.cu_seqlens, a.H, a.total);
    trace_end(TR_BWD_PRE, st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // d = 64 and 128: the TMEM-resident kernels of fa_bwd128.cu; d = 32: the kernels below
  if constexpr (D == 128 || D == 64) {
    return launch_bwd128(a, D, BF16, CAUSAL, st);
  } else {
  {
    auto kern = dkdv_kernel<D, BF16, CAUSAL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DkdvCfg<D>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const long long grid = static_cast<long long>(nqb) * (a.BH / a.group);   // per K/V head
    trace_begin(TR_BWD_DKDV, st);
    kern<<<static_cast<unsigned>(grid), THREADS, DkdvCfg<D>::SMEM_BYTES, st>>>(
        a.tmQ, a.tmK, a.tmV, a.tmdO, a.Dvec, Lp, a.dK, a.dV, a.N, Np, a.group, a.window,
        a.cu_seqlens, a.H, a.total, a.scale, a.c_log2, a.ctl);
    trace_end(TR_BWD_DKDV, st);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  {
    auto kern = dq_kernel<D, BF16, CAUSAL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DqCfg<D>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const long long grid = static_cast<long long>(nqb) * a.BH;
    trace_begin(TR_BWD_DQ, st);
    kern<<<static_cast<unsigned>(grid), THREADS, DqCfg<D>::SMEM_BYTES, st>>>(
        a.tmQ, a.tmK, a.tmV, a.tmdO, a.Dvec, Lp, a.dQ, a.N, Np, a.group, a.window, a.cu_seqlens,
        a.H, a.total, a.scale, a.c_log2, a.ctl);
    trace_end(TR_BWD_DQ, st);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
  }
}

}  // namespace

size_t bwd_workspace_bytes(long long BH, int N, int /*d*/) {
  const long long Np = static_cast<long long>((N + BM - 1) / BM) * BM;
  return static_cast<size_t>(2 * BH * Np) * sizeof(float);
}

cudaError_t launch_bwd(const BwdArgs& a, int d, bool bf16, bool causal, cudaStream_t st) {
#define FA_BWD_CASE(DD, BB, CC) \
  if (d == DD && bf16 == BB && causal == CC) return launch_bwd_t<DD, BB, CC>(a, st);
  FA_BWD_CASE(32, false, false) FA_BWD_CASE(32, false, true)
  FA_BWD_CASE(32, true, false) FA_BWD_CASE(32, true, true)
  FA_BWD_CASE(64, false, false) FA_BWD_CASE(64, false, true)
  FA_BWD_CASE(64, true, false) FA_BWD_CASE(64, true, true)
  FA_BWD_CASE(128, false, false) FA_BWD_CASE(128, false, true)
  FA_BWD_CASE(128, true, false) FA_BWD_CASE(128, true, true)
#undef FA_BWD_CASE
  return cudaErrorInvalidValue;
}

}  // namespace fa
