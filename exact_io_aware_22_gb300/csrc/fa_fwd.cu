// fa_fwd.cu -- exact attention forward (FlashAttention-2 order) for sm_103a.
//
// Method: "flash-attn-triton" docs page, sections "Tiling softmax is exact
// algebra" and Fig. 3 (running max m, running sum l, correction alpha applied to
// l and the accumulator together, one divide after the loop, L = m + log l, exp2
// with log2(e) folded into the scale), "Scope" (Q in the outer loop, grid split
// over the sequence, causal mask only on diagonal tiles, ragged N), and Fig. 1
// (one program per BLOCK_M query rows, K/V streamed BLOCK_N at a time).
//
// GB300 mapping (one CTA per SM, 384 threads):
//   warp 0      TMA producer: both Q tiles once, then K_j / V_j into a ring.
//   warp 1      TMEM allocator; lane 0 issues every tcgen05.mma and commit.
//   warps 4-7   softmax warpgroup for Q tile 0 (one thread per query row).
//   warps 8-11  softmax warpgroup for Q tile 1.
// TMEM (512 columns): S0 | S1 | O0 | O1.  S_t = Q_t K_j^T lands in fp32; the
// softmax thread of a row reads its 128 scores, writes P back over the first 64
// columns of S_t as packed 16-bit pairs, and the P.V MMA reads P straight from
// TMEM (A operand in tensor memory).  MMA issue order per K/V tile j is
//   PV0(j), S0(j+1), PV1(j), S1(j+1)
// so each softmax warpgroup overlaps two MMAs of the other tile.
//
// Running max update is lazy: m only moves when the tile maximum exceeds it by
// more than RESCALE_LOG2 (log2 units), so the O rescale (TMEM load-multiply-
// store) is skipped on almost every tile.  The result is still exact algebra:
// numerator and denominator carry the same stale m, and every p <= 2^8.
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

namespace {

constexpr int BM = 128;       // query rows per Q tile (= TMEM lanes)
constexpr int BN = 128;       // keys per K/V tile
constexpr int NT = 2;         // Q tiles per CTA
constexpr int THREADS = 384;
constexpr float RESCALE_LOG2 = 8.0f;

template <int D>
struct Cfg {
  static constexpr int STAGES = D == 128 ? 2 : 3;
  static constexpr int SW = D == 32 ? 64 : 128;        // swizzle width in bytes
  static constexpr int ATOM = SW / 2;                  // elements per swizzled row
  static constexpr int NCHUNK = D / ATOM;              // swizzle-width column blocks per tile
  static constexpr int CHUNK_BYTES = 128 * SW;         // one column block of a 128-row tile
  static constexpr int TILE_BYTES = 128 * D * 2;
  static constexpr uint32_t SWZ = D == 32 ? UMMA_SW64 : UMMA_SW128;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + NT * TILE_BYTES;
  static constexpr int V_OFF = K_OFF + STAGES * TILE_BYTES;
  static constexpr int BAR_OFF = V_OFF + STAGES * TILE_BYTES;
  // q_full, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2], p_full[2], o_full[2], done
  static constexpr int NBARS = 1 + 4 * STAGES + 7;
  static constexpr int SLOT_OFF = BAR_OFF + NBARS * 8;
  static constexpr int SMEM_BYTES = SLOT_OFF + 16 + 1024;   // + alignment slack
  static constexpr int TMEM_COLS = 512;
  static constexpr int S_COL = 0;                           // S_t at t * 128
  static constexpr int O_COL = 256;                         // O_t at 256 + t * D
};

// byte offset of k-step kk (16 elements along K) inside a K-major tile
template <int D>
__device__ __forceinline__ uint32_t kmajor_koff(int kk) {
  using C = Cfg<D>;
  const int e = kk * 16;
  return (e / C::ATOM) * C::CHUNK_BYTES + (e % C::ATOM) * 2;
}

template <int D, bool BF16, bool CAUSAL, bool WINDOW, bool PACKED>
__global__ void __launch_bounds__(THREADS, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, void* __restrict__ Out,
               float* __restrict__ Lout, int N, int n_qblk, int group, int window,
               const int* __restrict__ cu_seqlens, int H, int total, float c_log2,
               KernelCtl ctl) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* sg = smem_raw + (sb - raw);

  grid_dep_launch();                            // the next kernel may start setting up
  if constexpr (PACKED) grid_dep_wait();        // the offsets may come from earlier work
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BlockPos bp = block_pos(n_qblk);
  const int bh = bp.bh;
  const int qblk = n_qblk - 1 - bp.rank;        // causal: the last query tiles have the most work
  const int bkv = bh / group;                   // the K/V head of this query head (b-major heads)
  // Rows of this (batch, head): dense (B, H, N, d) maps are (d, N, B*H), a row at
  // (row, flat head); packed sequences (total, H, d) have maps (d, H, total), a row at
  // (head within the batch, first token + row), and their own length Nr.
  const SeqRows sr = seq_rows_t<PACKED>(cu_seqlens, bh / H, N, total);
  const int Nr = sr.n;
  const int hq = sr.packed ? bh % H : bh, hk = sr.packed ? (bh % H) / group : bkv;
  auto cy = [&](int r, int head) { return sr.y(r, head); };
  auto cz = [&](int r, int head) { return sr.z(r, head); };
  const int row0 = qblk * (NT * BM);
  const int nkv = (Nr + BN - 1) / BN;
  // KV tiles [lo_t[t], n_t[t]) of Q tile t: up to the diagonal when causal; with a
  // sliding window of W keys, from the tile holding key (first row - W + 1)
  int n_t[NT], lo_t[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int r = row0 + t * BM;
    if (r >= Nr) n_t[t] = 0;
    else if (CAUSAL) n_t[t] = min(nkv, min(r + BM - 1, Nr - 1) / BN + 1);
    else n_t[t] = nkv;
    lo_t[t] = WINDOW ? max(0, r - window + 1) / BN : 0;
  }
  const int j0 = lo_t[0];                       // the stream starts at tile 0's first KV tile
  const int n_max = max(n_t[0], n_t[1]);
  const int n_stream = n_max - j0;              // KV tiles loaded, j0 .. n_max - 1
  if (n_stream <= 0) return;                    // query tiles past the end of a packed sequence

  auto bar = [&](int i) -> uint32_t { return sb + C::BAR_OFF + 8 * i; };
  const int B_QF = 0;
  auto B_KF = [&](int s) { return 1 + s; };
  auto B_KE = [&](int s) { return 1 + C::STAGES + s; };
  auto B_VF = [&](int s) { return 1 + 2 * C::STAGES + s; };
  auto B_VE = [&](int s) { return 1 + 3 * C::STAGES + s; };
  auto B_SF = [&](int t) { return 1 + 4 * C::STAGES + t; };
  auto B_PF = [&](int t) { return 3 + 4 * C::STAGES + t; };
  auto B_OF = [&](int t) { return 5 + 4 * C::STAGES + t; };
  const int B_DONE = 7 + 4 * C::STAGES;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBARS; ++i) mbar_init(bar(i), 1);
    for (int t = 0; t < NT; ++t) mbar_init(bar(B_PF(t)), 128);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sb + C::SLOT_OFF, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sg + C::SLOT_OFF);
  grid_dep_wait();                              // inputs written, outputs free to overwrite

  if (warp == 0) {
    regs_dec<kRegsLow>();                          // warpgroup 0 (TMA, MMA issue): few registers
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_stream > 0) {
      bool ok = true;
      mbar_arrive_expect_tx(bar(B_QF), NT * C::TILE_BYTES);
      for (int t = 0; t < NT; ++t)
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d(sb + C::Q_OFF + t * C::TILE_BYTES + c * C::CHUNK_BYTES, &tmQ, bar(B_QF),
                      c * C::ATOM, cy(row0 + t * BM, hq), cz(row0 + t * BM, hq));
      int j = 0;                                // stream position: KV tile j0 + j
      for (; j < n_stream; ++j) {
        const int s = j % C::STAGES;
        const uint32_t ph = (j / C::STAGES) & 1;
        const int krow = (j0 + j) * BN;
        if (!(ok = mbar_wait(bar(B_KE(s)), ph ^ 1, ctl))) break;
        mbar_arrive_expect_tx(bar(B_KF(s)), C::TILE_BYTES);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d(sb + C::K_OFF + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &tmK, bar(B_KF(s)),
                      c * C::ATOM, cy(krow, hk), cz(krow, hk));
        if (!(ok = mbar_wait(bar(B_VE(s)), ph ^ 1, ctl))) { ++j; break; }
        mbar_arrive_expect_tx(bar(B_VF(s)), C::TILE_BYTES);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d(sb + C::V_OFF + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &tmV, bar(B_VF(s)),
                      c * C::ATOM, cy(krow, hk), cz(krow, hk));
      }
      if (!ok) {
        // drain: wait (bounded) for every copy this thread issued, so no bulk
        // copy lands in shared memory after the CTA has gone.
        mbar_wait(bar(B_QF), 0, ctl);
        for (int jj = max(0, j - C::STAGES); jj < j; ++jj) {
          const int s = jj % C::STAGES;
          const uint32_t ph = (jj / C::STAGES) & 1;
          mbar_wait(bar(B_KF(s)), ph, ctl);
          mbar_wait(bar(B_VF(s)), ph, ctl);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    regs_dec<kRegsLow>();
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_stream > 0) {
      constexpr uint32_t idS = umma_idesc_f16(BM, BN, BF16, false, false);
      constexpr uint32_t idO = umma_idesc_f16(BM, D, BF16, false, true);
      // descriptor low words of Q tile 0 and of stage 0 of the K and V rings (K-major
      // with LBO 16; V MN-major with LBO = one swizzle-width chunk); tiles and stages
      // are TILE_BYTES apart
      constexpr uint32_t HI = sdesc_hi(8 * C::SW, C::SWZ), STAGE_W = C::TILE_BYTES >> 4;
      const uint32_t q_lo = sdesc_lo(sb + C::Q_OFF, 16), k_lo = sdesc_lo(sb + C::K_OFF, 16);
      const uint32_t v_lo = sdesc_lo(sb + C::V_OFF, C::CHUNK_BYTES);
      auto issue_S = [&](int t, int s) {
        const uint32_t qa = q_lo + t * STAGE_W, ka = k_lo + s * STAGE_W;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = kmajor_koff<D>(kk) >> 4;
          umma_ss_w(tmem + C::S_COL + t * BN, qa + o, ka + o, HI, idS, kk > 0);
        }
      };
      auto issue_PV = [&](int t, int s, bool acc) {
        const uint32_t va = v_lo + s * STAGE_W, acc0 = acc ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          umma_ts_w(tmem + C::O_COL + t * D, tmem + C::S_COL + t * BN + kk * 8,
                    va + ((kk * 16 * C::SW) >> 4), HI, idO, kk > 0 ? 1u : acc0);
        }
      };
      bool ok = mbar_wait(bar(B_QF), 0, ctl) && mbar_wait(bar(B_KF(0)), 0, ctl);
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < NT; ++t)
          if (lo_t[t] == j0 && n_t[t] > j0) {
            issue_S(t, 0);
            umma_commit(bar(B_SF(t)));
          }
        umma_commit(bar(B_KE(0)));
      }
      // stream position jj holds KV tile j = j0 + jj; Q tile t takes part while
      // lo_t[t] <= j < n_t[t], its own iteration index being j - lo_t[t]
      for (int jj = 0; ok && jj < n_stream; ++jj) {
        const int j = j0 + jj;
        const int s = jj % C::STAGES;
        const int s1 = (jj + 1) % C::STAGES;
        const uint32_t ph = (jj / C::STAGES) & 1, ph1 = ((jj + 1) / C::STAGES) & 1;
        if (!(ok = mbar_wait(bar(B_VF(s)), ph, ctl))) break;
        bool k_next = false;
        for (int t = 0; t < NT && ok; ++t) {
          const bool in_t = j >= lo_t[t] && j < n_t[t];
          if (in_t) {
            if (!(ok = mbar_wait(bar(B_PF(t)), (j - lo_t[t]) & 1, ctl))) break;
            tc_fence_after();
            issue_PV(t, s, j > lo_t[t]);
          }
          if (j + 1 >= lo_t[t] && j + 1 < n_t[t]) {
            if (!k_next) {
              if (!(ok = mbar_wait(bar(B_KF(s1)), ph1, ctl))) break;
              tc_fence_after();
              k_next = true;
            }
            issue_S(t, s1);
            umma_commit(bar(B_SF(t)));
          } else if (in_t) {
            umma_commit(bar(B_OF(t)));
          }
        }
        if (!ok) break;
        umma_commit(bar(B_VE(s)));
        if (k_next) umma_commit(bar(B_KE(s1)));
      }
      // every MMA this thread issued has completed before TMEM is released
      umma_commit(bar(B_DONE));
      mbar_wait(bar(B_DONE), 0, ctl);
    }
    __syncwarp();
  } else if (warp >= 4) {
    regs_inc<kRegsHigh>();                         // the compute warpgroups take what it gives back
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;
    const int rit = (warp & 3) * 32 + lane;              // row within the tile (= TMEM lane)
    const int grow = row0 + t * BM + rit;                // query row
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::S_COL + t * BN;
    const uint32_t tO = tmem + lane_off + C::O_COL + t * D;
    const int nt = n_t[t] - lo_t[t];             // this tile's KV tiles, from lo_t[t]
    const int tile_row0 = row0 + t * BM;
    const int lo_key = WINDOW ? grow - window + 1 : 0;   // first allowed key
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      if (!(ok = mbar_wait_warp(bar(B_SF(t)), j & 1, ctl))) break;
      tc_fence_after();
      uint32_t sr[BN];
      tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
      tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
      tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
      tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
      const int kbase = (lo_t[t] + j) * BN;
      // masks: causal on the diagonal tile, key padding on the last tile, and with a
      // window the tiles reaching left of some row's first allowed key
      const bool need_mask = (CAUSAL && kbase + BN - 1 > tile_row0) || (kbase + BN > Nr) ||
                             (WINDOW && kbase < tile_row0 + BM - window);
      if (need_mask) {
        const int lim = CAUSAL ? min(grow + 1, Nr) : Nr;   // keys in [lo_key, lim) are allowed
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (kbase + c >= lim || (WINDOW && kbase + c < lo_key)) sr[c] = __float_as_uint(-INFINITY);
      }
      // row maximum: four independent chains of 3-input max
      const float mx = row_max128(sr);
      const float m_tile = mx * c_log2;
      const bool grow_m = m_tile > m_run + RESCALE_LOG2;
      const float m_use = grow_m ? m_tile : m_run;
      const float alpha = grow_m ? ex2(m_run - m_use) : 1.f;
      const float m_sub = (m_use == -INFINITY) ? 0.f : m_use;
      const float2 c2 = make_float2(c_log2, c_log2), nm2 = make_float2(-m_sub, -m_sub);
      float2 rs2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = 32 * h + 2 * i;
          const float2 t = fma2(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), c2, nm2);
          const float2 pp = make_float2(ex2(t.x), ex2(t.y));
          rs2[i & 1] = add2(rs2[i & 1], pp);
          pk[i] = pack2<BF16>(pp.x, pp.y);
        }
        tmem_st16(tS + 16 * h, pk);
      }
      const float rs = (rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y);
      l_run = l_run * alpha + rs;
      if (j > 0 && __any_sync(0xffffffffu, grow_m)) {
        // O holds sum over tiles < j; PV(j-1) has completed because S(j) was
        // issued after it and its commit was observed above.
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * cc, o);
          tmem_ld_wait_regs(o);
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 v = mul2(make_float2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), a2);
            o[2 * i] = __float_as_uint(v.x);
            o[2 * i + 1] = __float_as_uint(v.y);
          }
          tmem_st32(tO + 32 * cc, o);
        }
      }
      m_run = m_use;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(B_PF(t)));
    }
    if (ok && nt > 0 && mbar_wait_warp(bar(B_OF(t)), 0, ctl)) {
      tc_fence_after();
      const float inv_l = 1.f / l_run;
      const bool valid = grow < Nr;
      using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
      T* orow = reinterpret_cast<T*>(Out) + sr.off(grow, hq, H, N, D);
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * cc, o);
        tmem_ld_wait_regs(o);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l,
                             __uint_as_float(o[2 * i + 1]) * inv_l);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * cc);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      if (valid)
        Lout[sr.packed ? static_cast<size_t>(hq) * total + sr.base + grow
                       : static_cast<size_t>(bh) * N + grow] =
            (m_run + log2f(l_run)) * 0.69314718055994531f;
    }
  } else {
    regs_dec<kRegsLow>();                          // warps 2 and 3: idle
  }
  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool BF16, bool CAUSAL, bool WINDOW, bool PACKED>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t st) {
  using C = Cfg<D>;
  auto kern = fwd_kernel<D, BF16, CAUSAL, WINDOW, PACKED>;
  cudaError_t e = check_split_regs(reinterpret_cast<const void*>(kern));
  if (e != cudaSuccess) return e;
  e = ensure_smem(reinterpret_cast<const void*>(kern), C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int n_qblk = (a.N + NT * BM - 1) / (NT * BM);
  const long long grid = static_cast<long long>(n_qblk) * a.BH;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  trace_begin(TR_FWD, st);
  e = launch_dependent(kern, static_cast<unsigned>(grid), THREADS, C::SMEM_BYTES, st, a.tmQ,
                       a.tmK, a.tmV, a.O, a.L, a.N, n_qblk, a.group, a.window, a.cu_seqlens, a.H,
                       a.total, a.c_log2, a.ctl);
  trace_end(TR_FWD, st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// ============================================================== head dim <= 64
// At d <= 64 one 128-row query tile at a time per CTA, two CTAs per SM, and each
// CTA persistent.  A single issuing thread starts one tcgen05.mma about every 46
// cycles, which is what an M = 128, N <= 64 product (P.V at these head dims) needs at
// full rate only when two threads issue side by side; two resident CTAs also keep the
// tensor pipe and the exponential unit busy while the other waits.  A CTA starts with
// the tile of its own index and then takes further tiles from CTAs that have not been
// launched yet (cluster launch control), so the set-up (barriers, TMEM) is paid once
// per CTA, the next tile's Q and K/V loads overlap the end of the current tile, and
// the grid's longest-first order still decides which tile comes next.
//   warp 0      TMA producer and scheduler: publishes each tile in a two-slot ring,
//               loads its Q tile (double-buffered) and streams K_j / V_j into a ring
//               that runs on across tiles, then asks for the next tile.
//   warp 1      TMEM allocator; lane 0 issues every tcgen05.mma and commit.
//   warps 2-5   softmax, one thread per query row (TMEM lane quadrant = warp % 4),
//               and the epilogue of each tile.
// TMEM (256 columns): S (128 fp32) | P (64: 128 keys as 16-bit pairs) | O (d fp32).
// P has columns of its own, so S(g+1) is issued as soon as the softmax threads hold
// S(g), and runs under their exponentials; P.V(g) then runs under softmax(g+1), which
// waits for it only before storing P(g+1) (and before an O rescale).  The step index
// g runs on across tiles, so the MMA issue order is S(0), S(1), PV(0), S(2), PV(1), ...
// whatever tile each step belongs to.  The first P.V of a tile overwrites O; the
// softmax threads arrive on p_full only after their epilogue has read the previous
// tile's O out of TMEM, so that order is kept without a barrier of its own.
namespace one {
constexpr int THREADS = 192;
template <int D>
struct Cfg1 {
  using C = Cfg<D>;                                         // swizzle geometry of a tile
  static constexpr int STAGES = D == 64 ? 2 : 4;
  static constexpr int TILE_BYTES = C::TILE_BYTES;
  static constexpr int Q_OFF = 0;                           // two Q buffers
  static constexpr int K_OFF = 2 * TILE_BYTES;
  static constexpr int V_OFF = K_OFF + STAGES * TILE_BYTES;
  static constexpr int O_OFF = V_OFF + STAGES * TILE_BYTES;   // O rows staged for the store
  static constexpr int BAR_OFF = O_OFF + TILE_BYTES;
  // q_full[2], q_empty[2], k_full[S], k_empty[S], v_full[S], v_empty[S], s_full, s_free,
  // p_full, pv_done, o_full, done, tile_full[2], tile_empty[2], clc
  static constexpr int NBARS = 4 + 4 * STAGES + 6 + 5;
  static constexpr int CLC_OFF = (BAR_OFF + NBARS * 8 + 15) / 16 * 16;   // 16-byte response
  static constexpr int SLOT_OFF = CLC_OFF + 16;             // TMEM base, tile slots[2]
  static constexpr int SMEM_BYTES = SLOT_OFF + 16;
  static constexpr int TMEM_COLS = 256;
  static constexpr uint32_t S_COL = 0, P_COL = 128, O_COL = 192;
  // two CTAs per SM, each with the 1 KiB the system reserves per CTA
  static_assert(2 * (SMEM_BYTES + 1024) <= 233472, "two CTAs per SM must fit");
  static_assert(O_COL + D <= TMEM_COLS, "TMEM layout");
};

// One query tile of the grid: which head and rows, and its KV tiles [lo, lo + nt).
struct Tile1 {
  int bh, hq, hk, row0, lo, nt;
  SeqRows sr;
};
template <bool CAUSAL, bool WINDOW, bool PACKED>
__device__ __forceinline__ Tile1 tile1(int id, int n_qt, int N, int group, int window,
                                       const int* __restrict__ cu_seqlens, int H, int total) {
  Tile1 t;
  const BlockPos bp = block_pos(n_qt, id);
  t.bh = bp.bh;
  const int qt = n_qt - 1 - bp.rank;            // causal: the last query tiles have the most work
  t.sr = seq_rows_t<PACKED>(cu_seqlens, t.bh / H, N, total);
  const int Nr = t.sr.n;
  t.hq = t.sr.packed ? t.bh % H : t.bh;
  t.hk = t.sr.packed ? (t.bh % H) / group : t.bh / group;
  t.row0 = qt * BM;
  // up to the diagonal when causal; with a sliding window of W keys, from the tile
  // holding key (first row - W + 1); none for a tile past the end of a packed sequence
  const int nkv = (Nr + BN - 1) / BN;
  const int hi = CAUSAL ? min(nkv, min(t.row0 + BM - 1, Nr - 1) / BN + 1) : nkv;
  t.lo = WINDOW ? max(0, t.row0 - window + 1) / BN : 0;
  t.nt = t.row0 >= Nr ? 0 : hi - t.lo;
  return t;
}
}  // namespace one

template <int D, bool BF16, bool CAUSAL, bool WINDOW, bool PACKED>
__global__ void __launch_bounds__(one::THREADS, 2)
    fwd1_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, void* __restrict__ Out,
                float* __restrict__ Lout, int N, int n_qt, int group, int window,
                const int* __restrict__ cu_seqlens, int H, int total, float c_log2,
                KernelCtl ctl) {
  using C = Cfg<D>;
  using C1 = one::Cfg1<D>;
  constexpr int STAGES = C1::STAGES;
  extern __shared__ __align__(1024) uint8_t sg[];
  const uint32_t sb = smem_u32(sg);
  grid_dep_launch();                            // the next kernel may start setting up
  if (sb & 1023u) {                             // see FA_DEV_SMEM_ALIGN
    grid_dep_wait();
    if (threadIdx.x == 0) atomicOr(ctl.status, FA_DEV_SMEM_ALIGN);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto tile_of = [&](int id) {
    return one::tile1<CAUSAL, WINDOW, PACKED>(id, n_qt, N, group, window, cu_seqlens, H, total);
  };

  auto bar = [&](int i) -> uint32_t { return sb + C1::BAR_OFF + 8 * i; };
  auto B_QF = [&](int b) { return b; };
  auto B_QE = [&](int b) { return 2 + b; };
  auto B_KF = [&](int st) { return 4 + st; };
  auto B_KE = [&](int st) { return 4 + STAGES + st; };
  auto B_VF = [&](int st) { return 4 + 2 * STAGES + st; };
  auto B_VE = [&](int st) { return 4 + 3 * STAGES + st; };
  const int B_SF = 4 + 4 * STAGES, B_SFREE = B_SF + 1, B_PF = B_SF + 2, B_PVD = B_SF + 3,
            B_OF = B_SF + 4, B_DONE = B_SF + 5;
  auto B_TF = [&](int b) { return B_SF + 6 + b; };
  auto B_TE = [&](int b) { return B_SF + 8 + b; };
  const int B_CLC = B_SF + 10;
  volatile int* slot = reinterpret_cast<volatile int*>(sg + C1::SLOT_OFF + 4);
  const uint32_t clc_resp = sb + C1::CLC_OFF;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C1::NBARS; ++i) mbar_init(bar(i), 1);
    mbar_init(bar(B_SFREE), 128);
    mbar_init(bar(B_PF), 128);
    mbar_init(bar(B_TE(0)), 5);                 // the MMA thread and one lane per softmax warp
    mbar_init(bar(B_TE(1)), 5);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sb + C1::SLOT_OFF, C1::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sg + C1::SLOT_OFF);
  grid_dep_wait();                              // inputs written, outputs free to overwrite

  // Consumers read tile k from slot k & 1; the last tile published is -1.
  auto next_tile = [&](int k, bool& ok) -> int {
    if (!(ok = mbar_wait(bar(B_TF(k & 1)), (k >> 1) & 1, ctl))) return -1;
    return slot[k & 1];
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer, scheduler
    if (lane == 0) {
      bool ok = true;
      int tile = static_cast<int>(blockIdx.x);
      int g = 0, kq = 0, nk = 0, nv = 0;         // steps, Q tiles, K and V tiles loaded
      bool pending = false;                       // a request for the next tile is out
      int n_req = 0;                               // requests made
      for (int k = 0; ok; ++k) {
        if (!(ok = mbar_wait(bar(B_TE(k & 1)), ((k >> 1) & 1) ^ 1, ctl))) break;
        slot[k & 1] = tile;
        mbar_arrive(bar(B_TF(k & 1)));          // release: the slot write is seen with the phase
        if (tile < 0) break;
        // ask for the next tile together with this tile's last loads: early enough that
        // the answer is there when they complete, late enough that a CTA takes a tile
        // only when it is nearly free (asking at a tile's start handed the last tiles to
        // CTAs that still had most of a long tile ahead, and took tiles from CTAs that had
        // not started yet when all would have fit at once)
        auto request = [&]() {
          mbar_arrive_expect_tx(bar(B_CLC), 16);
          clc_try_cancel(clc_resp, bar(B_CLC));
          pending = true;
          ++n_req;
        };
        const one::Tile1 t = tile_of(tile);
        if (t.nt <= 0) request();
        if (t.nt > 0) {
          const int qb = kq & 1;
          if (!(ok = mbar_wait(bar(B_QE(qb)), ((kq >> 1) & 1) ^ 1, ctl))) break;
          mbar_arrive_expect_tx(bar(B_QF(qb)), C1::TILE_BYTES);
          for (int c = 0; c < C::NCHUNK; ++c)
            tma_load_3d(sb + C1::Q_OFF + qb * C1::TILE_BYTES + c * C::CHUNK_BYTES, &tmQ,
                        bar(B_QF(qb)), c * C::ATOM, t.sr.y(t.row0, t.hq), t.sr.z(t.row0, t.hq));
          ++kq;
          for (int j = 0; j < t.nt; ++j, ++g) {
            const int st = g % STAGES;
            const uint32_t ph = (g / STAGES) & 1;
            const int krow = (t.lo + j) * BN;
            if (!(ok = mbar_wait(bar(B_KE(st)), ph ^ 1, ctl))) break;
            mbar_arrive_expect_tx(bar(B_KF(st)), C1::TILE_BYTES);
            for (int c = 0; c < C::NCHUNK; ++c)
              tma_load_3d(sb + C1::K_OFF + st * C1::TILE_BYTES + c * C::CHUNK_BYTES, &tmK,
                          bar(B_KF(st)), c * C::ATOM, t.sr.y(krow, t.hk), t.sr.z(krow, t.hk));
            ++nk;
            if (!(ok = mbar_wait(bar(B_VE(st)), ph ^ 1, ctl))) break;
            mbar_arrive_expect_tx(bar(B_VF(st)), C1::TILE_BYTES);
            for (int c = 0; c < C::NCHUNK; ++c)
              tma_load_3d(sb + C1::V_OFF + st * C1::TILE_BYTES + c * C::CHUNK_BYTES, &tmV,
                          bar(B_VF(st)), c * C::ATOM, t.sr.y(krow, t.hk), t.sr.z(krow, t.hk));
            ++nv;
            if (j + 1 == t.nt) request();
          }
          if (!ok) break;
        }
        // the next tile: a CTA that had not started, if any was left
        if (!(ok = mbar_wait(bar(B_CLC), k & 1, ctl))) break;
        pending = false;
        tile = clc_result(clc_resp);
      }
      if (!ok) {
        if (pending) mbar_wait(bar(B_CLC), (n_req - 1) & 1, ctl);   // the response lands in smem
        // drain: wait (bounded) for the copies this thread may still have in flight, so
        // no bulk copy lands in shared memory after the CTA has gone
        for (int i = max(0, kq - 2); i < kq; ++i) mbar_wait(bar(B_QF(i & 1)), (i >> 1) & 1, ctl);
        for (int i = max(0, nk - STAGES); i < nk; ++i)
          mbar_wait(bar(B_KF(i % STAGES)), (i / STAGES) & 1, ctl);
        for (int i = max(0, nv - STAGES); i < nv; ++i)
          mbar_wait(bar(B_VF(i % STAGES)), (i / STAGES) & 1, ctl);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = umma_idesc_f16(BM, BN, BF16, false, false);
      constexpr uint32_t idO = umma_idesc_f16(BM, D, BF16, false, true);
      constexpr uint32_t HI = sdesc_hi(8 * C::SW, C::SWZ), STAGE_W = C1::TILE_BYTES >> 4;
      const uint32_t q_lo = sdesc_lo(sb + C1::Q_OFF, 16), k_lo = sdesc_lo(sb + C1::K_OFF, 16);
      const uint32_t v_lo = sdesc_lo(sb + C1::V_OFF, C::CHUNK_BYTES);
      // the pending P.V: step, stage, whether it is its tile's first / last
      int pv_g = -1, pv_st = 0;
      bool pv_first = false, pv_last = false;
      bool ok = true;
      auto issue_pv = [&]() -> bool {
        if (!mbar_wait(bar(B_VF(pv_st)), (pv_g / STAGES) & 1, ctl)) return false;
        if (!mbar_wait(bar(B_PF), pv_g & 1, ctl)) return false;
        tc_fence_after();
        const uint32_t va = v_lo + pv_st * STAGE_W;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          umma_ts_w(tmem + C1::O_COL, tmem + C1::P_COL + kk * 8,
                    va + ((kk * 16 * C::SW) >> 4), HI, idO, (kk > 0 || !pv_first) ? 1u : 0u);
        umma_commit(bar(B_VE(pv_st)));
        umma_commit(bar(B_PVD));
        if (pv_last) umma_commit(bar(B_OF));
        return true;
      };
      int g = 0, kq = 0;
      for (int k = 0; ok; ++k) {
        const int tile = next_tile(k, ok);
        if (!ok) break;
        mbar_arrive(bar(B_TE(k & 1)));
        if (tile < 0) break;
        const one::Tile1 t = tile_of(tile);
        if (t.nt == 0) continue;
        const int qb = kq & 1;
        if (!(ok = mbar_wait(bar(B_QF(qb)), (kq >> 1) & 1, ctl))) break;
        const uint32_t qa = q_lo + qb * STAGE_W;
        for (int j = 0; j < t.nt; ++j, ++g) {
          // S(g) once K_g is in and the softmax threads hold S(g - 1)
          const int st = g % STAGES;
          if (!(ok = mbar_wait(bar(B_KF(st)), (g / STAGES) & 1, ctl))) break;
          if (g > 0 && !(ok = mbar_wait(bar(B_SFREE), (g - 1) & 1, ctl))) break;
          tc_fence_after();
          const uint32_t ka = k_lo + st * STAGE_W;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t o = kmajor_koff<D>(kk) >> 4;
            umma_ss_w(tmem + C1::S_COL, qa + o, ka + o, HI, idS, kk > 0);
          }
          umma_commit(bar(B_SF));
          umma_commit(bar(B_KE(st)));
          if (j + 1 == t.nt) umma_commit(bar(B_QE(qb)));   // Q free once its last S is done
          // then P(g - 1).V
          if (pv_g >= 0 && !(ok = issue_pv())) break;
          pv_g = g;
          pv_st = st;
          pv_first = j == 0;
          pv_last = j + 1 == t.nt;
        }
        // the tile's last P.V goes out before this thread waits for the next tile, so
        // the epilogue never waits on the next tile's loads
        if (ok && pv_g >= 0) ok = issue_pv();
        pv_g = -1;
        ++kq;
      }
      // every MMA this thread issued has completed before TMEM is released
      umma_commit(bar(B_DONE));
      mbar_wait(bar(B_DONE), 0, ctl);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax, epilogue
    const int rit = (warp & 3) * 32 + lane;      // row within the tile (= TMEM lane)
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C1::S_COL;
    const uint32_t tP = tmem + lane_off + C1::P_COL;
    const uint32_t tO = tmem + lane_off + C1::O_COL;
    bool ok = true;
    int g = 0, kq = 0;
    for (int k = 0; ok; ++k) {
      int tile = next_tile(k, ok);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_TE(k & 1)));
      if (tile < 0) break;
      const one::Tile1 t = tile_of(tile);
      if (t.nt == 0) continue;
      const int Nr = t.sr.n;
      const int grow = t.row0 + rit;             // query row
      const int lo_key = WINDOW ? grow - window + 1 : 0;   // first allowed key
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < t.nt; ++j, ++g) {
        if (!(ok = mbar_wait_warp(bar(B_SF), g & 1, ctl))) break;
        tc_fence_after();
        uint32_t sr_[BN];
        tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr_[0]));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr_[32]));
        tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr_[64]));
        tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr_[96]));
        tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&sr_[0]));
        tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&sr_[32]));
        tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&sr_[64]));
        tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&sr_[96]));
        tc_fence_before();
        mbar_arrive(bar(B_SFREE));               // S may now receive the next step
        const int kbase = (t.lo + j) * BN;
        // masks: causal on the diagonal tile, key padding on the last tile, and with a
        // window the tiles reaching left of some row's first allowed key
        const bool need_mask = (CAUSAL && kbase + BN - 1 > t.row0) || (kbase + BN > Nr) ||
                               (WINDOW && kbase < t.row0 + BM - window);
        if (need_mask) {
          const int lim = CAUSAL ? min(grow + 1, Nr) : Nr;   // keys in [lo_key, lim) are allowed
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (kbase + c >= lim || (WINDOW && kbase + c < lo_key)) sr_[c] = __float_as_uint(-INFINITY);
        }
        const float mx = row_max128(sr_);
        const float m_tile = mx * c_log2;
        const bool grow_m = m_tile > m_run + RESCALE_LOG2;
        const float m_use = grow_m ? m_tile : m_run;
        const float alpha = grow_m ? ex2(m_run - m_use) : 1.f;
        const float m_sub = (m_use == -INFINITY) ? 0.f : m_use;
        const float2 c2 = make_float2(c_log2, c_log2), nm2 = make_float2(-m_sub, -m_sub);
        float2 rs2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        // p for keys [32h, 32h + 32) as 16 packed pairs
        auto exp_pairs = [&](int h, uint32_t (&pk)[16]) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = 32 * h + 2 * i;
            const float2 tt = fma2(make_float2(__uint_as_float(sr_[c]), __uint_as_float(sr_[c + 1])),
                                   c2, nm2);
            const float2 pp = make_float2(ex2(tt.x), ex2(tt.y));
            rs2[i & 1] = add2(rs2[i & 1], pp);
            pk[i] = pack2<BF16>(pp.x, pp.y);
          }
        };
        // the first half of P before waiting for P(g-1).V; the second half is stored as
        // it is formed, so no more than half of P is held in registers
        uint32_t pa[16], pb[16];
        exp_pairs(0, pa);
        exp_pairs(1, pb);
        // P(g-1).V has completed: P's columns are free and O holds the sum over the
        // tile's earlier steps (at a tile's first step, the epilogue before it waited
        // for the previous tile's last P.V)
        if (j > 0) {
          if (!(ok = mbar_wait_warp(bar(B_PVD), (g - 1) & 1, ctl))) break;
          tc_fence_after();
        }
        tmem_st16(tP, pa);
        tmem_st16(tP + 16, pb);
        exp_pairs(2, pa);
        tmem_st16(tP + 32, pa);
        exp_pairs(3, pb);
        tmem_st16(tP + 48, pb);
        if (j > 0 && __any_sync(0xffffffffu, grow_m)) {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * cc, o);
            tmem_ld_wait_regs(o);
            const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 v = mul2(make_float2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), a2);
              o[2 * i] = __float_as_uint(v.x);
              o[2 * i + 1] = __float_as_uint(v.y);
            }
            tmem_st32(tO + 32 * cc, o);
          }
        }
        m_run = m_use;
        const float rs = (rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y);
        l_run = l_run * alpha + rs;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(B_PF));
      }
      if (!ok) break;
      // epilogue: O = acc / l and L once the tile's last P.V has completed
      if (!(ok = mbar_wait_warp(bar(B_OF), kq & 1, ctl))) break;
      ++kq;
      tc_fence_after();
      const float inv_l = 1.f / l_run;
      const bool valid = grow < Nr;
      // Each thread writes its row of O (16-bit) to this warp's 32 staging rows in shared
      // memory, 16-byte chunk c of row r at chunk c ^ (r mod CPR), so the eight lanes of
      // a store phase hit distinct banks; the warp then writes rows to global memory
      // 512 contiguous bytes per instruction.
      constexpr int CPR = D / 8;                 // 16-byte chunks per row
      uint4* stage = reinterpret_cast<uint4*>(sg + C1::O_OFF) + (warp & 3) * 32 * CPR;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * cc, o);
        tmem_ld_wait_regs(o);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l,
                             __uint_as_float(o[2 * i + 1]) * inv_l);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          stage[lane * CPR + ((4 * cc + i) ^ (lane % CPR))] =
              make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      }
      tc_fence_before();                         // O read before the next tile's p_full
      if (valid)
        Lout[t.sr.packed ? static_cast<size_t>(t.hq) * total + t.sr.base + grow
                         : static_cast<size_t>(t.bh) * N + grow] =
            (m_run + log2f(l_run)) * 0.69314718055994531f;
      __syncwarp();
      using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
      constexpr int RPI = 32 / CPR;              // rows per store instruction
#pragma unroll
      for (int i = 0; i < 32 / RPI; ++i) {
        const int r = i * RPI + lane / CPR, c = lane % CPR;   // row within the warp, chunk
        const int orow_g = t.row0 + (warp & 3) * 32 + r;
        if (orow_g < Nr) {
          T* dst = reinterpret_cast<T*>(Out) + t.sr.off(orow_g, t.hq, H, N, D) + 8 * c;
          *reinterpret_cast<uint4*>(dst) = stage[r * CPR + (c ^ (r % CPR))];
        }
      }
      __syncwarp();                              // staging rows free for the next tile
    }
  }
  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C1::TMEM_COLS);
  }
}

template <int D, bool BF16, bool CAUSAL, bool WINDOW, bool PACKED>
cudaError_t launch_fwd1_t(const FwdArgs& a, cudaStream_t st) {
  using C1 = one::Cfg1<D>;
  auto kern = fwd1_kernel<D, BF16, CAUSAL, WINDOW, PACKED>;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), C1::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int n_qt = (a.N + BM - 1) / BM;
  const long long grid = static_cast<long long>(n_qt) * a.BH;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  trace_begin(TR_FWD, st);
  e = launch_dependent(kern, static_cast<unsigned>(grid), one::THREADS, C1::SMEM_BYTES, st, a.tmQ,
                       a.tmK, a.tmV, a.O, a.L, a.N, n_qt, a.group, a.window, a.cu_seqlens, a.H,
                       a.total, a.c_log2, a.ctl);
  trace_end(TR_FWD, st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

FwdTileInfo fwd_tile_info(int d) {
  FwdTileInfo t;
  t.box_cols = d == 32 ? 32 : 64;
  t.box_rows = 128;
  t.swizzle_bytes = d == 32 ? 64 : 128;
  return t;
}

template <bool BF16, bool CAUSAL, bool WINDOW, bool PACKED>
cudaError_t launch_fwd_dd(const FwdArgs& a, int d, cudaStream_t st) {
  if (d == 32) return launch_fwd1_t<32, BF16, CAUSAL, WINDOW, PACKED>(a, st);
  if (d == 64) return launch_fwd1_t<64, BF16, CAUSAL, WINDOW, PACKED>(a, st);
  if (d == 128) return launch_fwd_t<128, BF16, CAUSAL, WINDOW, PACKED>(a, st);
  return cudaErrorInvalidValue;
}

template <bool BF16>
cudaError_t launch_fwd_b(const FwdArgs& a, int d, bool causal, bool window, bool packed,
                         cudaStream_t st) {
  if (!causal) return packed ? launch_fwd_dd<BF16, false, false, true>(a, d, st)
                             : launch_fwd_dd<BF16, false, false, false>(a, d, st);
  if (window) return packed ? launch_fwd_dd<BF16, true, true, true>(a, d, st)
                            : launch_fwd_dd<BF16, true, true, false>(a, d, st);
  return packed ? launch_fwd_dd<BF16, true, false, true>(a, d, st)
                : launch_fwd_dd<BF16, true, false, false>(a, d, st);
}

cudaError_t launch_fwd_d(const FwdArgs& a, int d, bool bf16, bool causal, bool window, bool packed,
                         cudaStream_t st) {
  return bf16 ? launch_fwd_b<true>(a, d, causal, window, packed, st)
              : launch_fwd_b<false>(a, d, causal, window, packed, st);
}

cudaError_t launch_fwd(const FwdArgs& a, int d, bool bf16, bool causal, cudaStream_t st) {
  // a sliding window is causal; windowed and packed-sequence kernels are separate
  // instantiations, so the plain dense ones carry none of their bookkeeping
  const bool window = causal && a.window > 0, packed = a.cu_seqlens != nullptr;
  return launch_fwd_d(a, d, bf16, causal, window, packed, st);
}

}  // namespace fa
