// fa_fwd8.cu -- attention forward on 8-bit E4M3 inputs (head dim 128) for sm_103a,
// and the E4M3 quantiser that prepares them.
//
// Method: as the 16-bit forward (fa_fwd.cu): the "flash-attn-triton" docs page,
// "Tiling softmax is exact algebra" and Fig. 3 (running max, running sum, alpha,
// one divide after the loop, exp2 with log2(e) folded into the scale), "Scope"
// (Q in the outer loop, causal mask only on diagonal tiles).  The inputs are in the
// FP8 precision that the FlashAttention note credits to FlashAttention-3 ("Versions
// and Evolution"), with per-tensor descale factors: the attention of q_scale Q,
// k_scale K and v_scale V.
//
// Both products run as tcgen05.mma kind::f8f6f4 with both operands K-major in
// shared memory, fp32 accumulators in TMEM:
//   S   = Q K^T     A = Q tile (128 rows x 128 bytes of d), B = K tile (same shape)
//   O  += P V       A = P (128 query rows x 128 keys as E4M3), written by the softmax
//                   threads into TMEM over the first 32 columns of their S tile (four
//                   codes per 32-bit column, the lowest key in the lowest byte); B =
//                   V^T tile (128 rows of d x 128 bytes of keys), V^T being the
//                   caller's transposed copy of V.
// At d = 128 every shared-memory tile is 128 rows of 128 bytes, one 128-byte swizzle
// span, so each product is four MMAs of K = 32 bytes.
//
// Warp roles and TMEM are those of the 16-bit forward (one CTA per SM, 384
// threads): warp 0 TMA, warp 1 TMEM and MMA issue, warps 4-7 / 8-11 softmax for
// query tiles 0 / 1; TMEM S0 | S1 | O0 | O1, P over the start of S as in the 16-bit
// forward: the S MMA of the next KV tile, which overwrites it, is issued after the
// P.V MMA that reads it, and the tensor pipe runs them in order.
// The probabilities p = 2^(s - m) lie in (0, 2^8] (lazy running max, as in the
// 16-bit forward), inside the E4M3 range (largest finite value 448); l sums the
// unrounded p.
#include "fa_internal.h"
#include "fa_ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>

namespace fa {

namespace {

constexpr int BM = 128;        // query rows per Q tile (= TMEM lanes)
constexpr int BN = 128;        // keys per K/V tile
constexpr int NT = 2;          // Q tiles per CTA
constexpr int HD = 128;        // head dim (bytes per Q/K row)
constexpr int THREADS = 384;
constexpr int STAGES = 3;
constexpr float RESCALE_LOG2 = 8.0f;

constexpr int TILE = 128 * 128;                 // one 128-row tile of 128 bytes
constexpr int Q_OFF = 0;
constexpr int K_OFF = Q_OFF + NT * TILE;
constexpr int V_OFF = K_OFF + STAGES * TILE;
constexpr int BAR_OFF = V_OFF + STAGES * TILE;
// q_full, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2], p_full[2], o_full[2], done
constexpr int NBARS = 1 + 4 * STAGES + 7;
constexpr int SLOT_OFF = BAR_OFF + NBARS * 8;
constexpr int SMEM_BYTES = SLOT_OFF + 16 + 1024;          // + alignment slack
constexpr int TMEM_COLS = 512;
constexpr int S_COL = 0;                                  // S_t at t * 128
constexpr int O_COL = 256;                                // O_t at 256 + t * 128

// Instruction descriptor, kind::f8f6f4: A and B both E4M3 (format 0), K-major,
// fp32 accumulator; N>>3 at bits 17..22, M>>4 at bits 24..28.
constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem], 8-bit operands, descriptors given as words.
__device__ __forceinline__ void umma8_ss_w(uint32_t d_tmem, uint32_t alo, uint32_t blo,
                                           uint32_t hi, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 a, b;\n\tmov.b64 a, {%1, %3};\n\tmov.b64 b, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a, b, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(alo), "r"(blo), "r"(hi), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], 8-bit operands (A: one row per lane, four codes per
// 32-bit column), B's descriptor given as words.
__device__ __forceinline__ void umma8_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint32_t blo,
                                           uint32_t hi, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 b;\n\tmov.b64 b, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], b, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(blo), "r"(hi), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE,
                                                        __NV_E4M3));
}

template <bool CAUSAL>
__global__ void __launch_bounds__(THREADS, 1)
    fwd8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmVt, __nv_bfloat16* __restrict__ Out,
                float* __restrict__ Lout, int N, int n_qblk, int group, float c_log2,
                float o_scale, KernelCtl ctl) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* sg = smem_raw + (sb - raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BlockPos bp = block_pos(n_qblk);
  const int bh = bp.bh;
  const int qblk = n_qblk - 1 - bp.rank;        // causal: the last query tiles have the most work
  const int bkv = bh / group;                   // the K/V head of this query head
  const int row0 = qblk * (NT * BM);
  const int nkv = (N + BN - 1) / BN;
  int n_t[NT];                                  // KV tiles [0, n_t) of Q tile t
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int r = row0 + t * BM;
    if (r >= N) n_t[t] = 0;
    else if (CAUSAL) n_t[t] = min(nkv, min(r + BM - 1, N - 1) / BN + 1);
    else n_t[t] = nkv;
  }
  const int n_stream = max(n_t[0], n_t[1]);

  auto bar = [&](int i) -> uint32_t { return sb + BAR_OFF + 8 * i; };
  const int B_QF = 0;
  auto B_KF = [&](int s) { return 1 + s; };
  auto B_KE = [&](int s) { return 1 + STAGES + s; };
  auto B_VF = [&](int s) { return 1 + 2 * STAGES + s; };
  auto B_VE = [&](int s) { return 1 + 3 * STAGES + s; };
  auto B_SF = [&](int t) { return 1 + 4 * STAGES + t; };
  auto B_PF = [&](int t) { return 3 + 4 * STAGES + t; };
  auto B_OF = [&](int t) { return 5 + 4 * STAGES + t; };
  const int B_DONE = 7 + 4 * STAGES;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBARS; ++i) mbar_init(bar(i), 1);
    for (int t = 0; t < NT; ++t) mbar_init(bar(B_PF(t)), 128);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sb + SLOT_OFF, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmVt);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sg + SLOT_OFF);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_stream > 0) {
      bool ok = true;
      mbar_arrive_expect_tx(bar(B_QF), NT * TILE);
      for (int t = 0; t < NT; ++t)
        tma_load_3d(sb + Q_OFF + t * TILE, &tmQ, bar(B_QF), 0, row0 + t * BM, bh);
      int j = 0;
      for (; j < n_stream; ++j) {
        const int s = j % STAGES;
        const uint32_t ph = (j / STAGES) & 1;
        if (!(ok = mbar_wait(bar(B_KE(s)), ph ^ 1, ctl))) break;
        mbar_arrive_expect_tx(bar(B_KF(s)), TILE);
        tma_load_3d(sb + K_OFF + s * TILE, &tmK, bar(B_KF(s)), 0, j * BN, bkv);
        if (!(ok = mbar_wait(bar(B_VE(s)), ph ^ 1, ctl))) { ++j; break; }
        mbar_arrive_expect_tx(bar(B_VF(s)), TILE);
        tma_load_3d(sb + V_OFF + s * TILE, &tmVt, bar(B_VF(s)), j * BN, 0, bkv);
      }
      if (!ok) {
        // drain: wait (bounded) for every copy this thread issued
        mbar_wait(bar(B_QF), 0, ctl);
        for (int jj = max(0, j - STAGES); jj < j; ++jj) {
          const int s = jj % STAGES;
          const uint32_t ph = (jj / STAGES) & 1;
          mbar_wait(bar(B_KF(s)), ph, ctl);
          mbar_wait(bar(B_VF(s)), ph, ctl);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_stream > 0) {
      constexpr uint32_t idS = idesc_e4m3(BM, BN);
      constexpr uint32_t idO = idesc_e4m3(BM, HD);
      // every operand: K-major, 128-byte swizzle, 8-row groups 1024 bytes apart; the
      // k-step of 32 bytes is +2 in the descriptor's low word
      constexpr uint32_t HI = sdesc_hi(1024, UMMA_SW128), TILE_W = TILE >> 4;
      const uint32_t q_lo = sdesc_lo(sb + Q_OFF, 16), k_lo = sdesc_lo(sb + K_OFF, 16);
      const uint32_t v_lo = sdesc_lo(sb + V_OFF, 16);
      auto issue_S = [&](int t, int s) {
        const uint32_t qa = q_lo + t * TILE_W, ka = k_lo + s * TILE_W;
#pragma unroll
        for (int kk = 0; kk < HD / 32; ++kk)
          umma8_ss_w(tmem + S_COL + t * BN, qa + 2 * kk, ka + 2 * kk, HI, idS, kk > 0);
      };
      auto issue_PV = [&](int t, int s, bool acc) {
        const uint32_t va = v_lo + s * TILE_W, acc0 = acc ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < BN / 32; ++kk)
          umma8_ts_w(tmem + O_COL + t * HD, tmem + S_COL + t * BN + 8 * kk, va + 2 * kk, HI, idO,
                     kk > 0 ? 1u : acc0);
      };
      bool ok = mbar_wait(bar(B_QF), 0, ctl) && mbar_wait(bar(B_KF(0)), 0, ctl);
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < NT; ++t)
          if (n_t[t] > 0) {
            issue_S(t, 0);
            umma_commit(bar(B_SF(t)));
          }
        umma_commit(bar(B_KE(0)));
      }
      for (int j = 0; ok && j < n_stream; ++j) {
        const int s = j % STAGES;
        const int s1 = (j + 1) % STAGES;
        const uint32_t ph = (j / STAGES) & 1, ph1 = ((j + 1) / STAGES) & 1;
        if (!(ok = mbar_wait(bar(B_VF(s)), ph, ctl))) break;
        bool k_next = false;
        for (int t = 0; t < NT && ok; ++t) {
          const bool in_t = j < n_t[t];
          if (in_t) {
            if (!(ok = mbar_wait(bar(B_PF(t)), j & 1, ctl))) break;
            tc_fence_after();
            issue_PV(t, s, j > 0);
          }
          if (j + 1 < n_t[t]) {
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
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;
    const int rit = (warp & 3) * 32 + lane;              // row within the tile (= TMEM lane)
    const int grow = row0 + t * BM + rit;                // query row
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + S_COL + t * BN;
    const uint32_t tO = tmem + lane_off + O_COL + t * HD;
    const int nt = n_t[t];
    const int tile_row0 = row0 + t * BM;
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
      const int kbase = j * BN;
      if ((CAUSAL && kbase + BN - 1 > tile_row0) || kbase + BN > N) {
        const int lim = CAUSAL ? min(grow + 1, N) : N;   // keys below lim are allowed
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (kbase + c >= lim) sr[c] = __float_as_uint(-INFINITY);
      }
      float mc[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        mc[q] = __uint_as_float(sr[32 * q]);
#pragma unroll
        for (int c = 1; c + 1 < 32; c += 2)
          mc[q] = fmax3(mc[q], __uint_as_float(sr[32 * q + c]), __uint_as_float(sr[32 * q + c + 1]));
        mc[q] = fmaxf(mc[q], __uint_as_float(sr[32 * q + 31]));
      }
      const float mx = fmaxf(fmax3(mc[0], mc[1], mc[2]), mc[3]);
      const float m_tile = mx * c_log2;
      const bool grow_m = m_tile > m_run + RESCALE_LOG2;
      const float m_use = grow_m ? m_tile : m_run;
      const float alpha = grow_m ? ex2(m_run - m_use) : 1.f;
      const float m_sub = (m_use == -INFINITY) ? 0.f : m_use;
      const float2 c2 = make_float2(c_log2, c_log2), nm2 = make_float2(-m_sub, -m_sub);
      float2 rs2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      uint32_t w[32];                            // the row of P: keys 4i .. 4i+3 in word i
#pragma unroll
      for (int h = 0; h < 4; ++h) {
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          const int c = 32 * h + 2 * i;
          const float2 t0 = fma2(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), c2, nm2);
          const float2 t1 = fma2(make_float2(__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])), c2, nm2);
          const float2 p0 = make_float2(ex2(t0.x), ex2(t0.y));
          const float2 p1 = make_float2(ex2(t1.x), ex2(t1.y));
          rs2[0] = add2(rs2[0], p0);
          rs2[1] = add2(rs2[1], p1);
          w[8 * h + i / 2] = e4m3x2(p0.x, p0.y) | (e4m3x2(p1.x, p1.y) << 16);
        }
      }
      tmem_st32(tS, w);                          // P over the first 32 columns of S
      const float rs = (rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y);
      l_run = l_run * alpha + rs;
      if (j > 0 && __any_sync(0xffffffffu, grow_m)) {
        // O holds the sum over tiles < j; PV(j-1) has completed because S(j) was
        // issued after it and its commit was observed above.
#pragma unroll
        for (int cc = 0; cc < HD / 32; ++cc) {
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
      const float mul = o_scale / l_run;
      const bool valid = grow < N;
      __nv_bfloat16* orow = Out + (static_cast<size_t>(bh) * N + grow) * HD;
#pragma unroll
      for (int cc = 0; cc < HD / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * cc, o);
        tmem_ld_wait_regs(o);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack2<true>(__uint_as_float(o[2 * i]) * mul, __uint_as_float(o[2 * i + 1]) * mul);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * cc);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      if (valid)
        Lout[static_cast<size_t>(bh) * N + grow] = (m_run + log2f(l_run)) * 0.69314718055994531f;
    }
  }
  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// E4M3 codes of x * inv_scale (round to nearest even, saturating at +-448), matrix
// by matrix; with TRANSPOSE the rows and columns of every matrix are swapped.
template <bool BF16>
__device__ __forceinline__ float in_f(const uint16_t* p) {
  return unpack2<BF16>(static_cast<uint32_t>(__ldg(p))).x;
}

template <bool BF16>
__global__ void __launch_bounds__(256)
    quant8_kernel(const uint16_t* __restrict__ X, uint8_t* __restrict__ Y, long long n,
                  float inv_scale) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride)
    Y[i] = static_cast<uint8_t>(
        __nv_cvt_float_to_fp8(in_f<BF16>(X + i) * inv_scale, __NV_SATFINITE, __NV_E4M3));
}

// 32 x 32 tiles through shared memory: block (32, 8), grid (col tiles, row tiles, mats).
template <bool BF16>
__global__ void __launch_bounds__(256)
    quant8_t_kernel(const uint16_t* __restrict__ X, uint8_t* __restrict__ Y, int rows, int cols,
                    float inv_scale) {
  __shared__ uint8_t tile[32][33];
  const size_t mat = static_cast<size_t>(blockIdx.z) * rows * cols;
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = r0 + ty + 8 * k, c = c0 + tx;
    if (r < rows && c < cols)
      tile[ty + 8 * k][tx] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(
          in_f<BF16>(X + mat + static_cast<size_t>(r) * cols + c) * inv_scale, __NV_SATFINITE,
          __NV_E4M3));
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int c = c0 + ty + 8 * k, r = r0 + tx;   // output row c (a column of X), column r
    if (r < rows && c < cols) Y[mat + static_cast<size_t>(c) * rows + r] = tile[tx][ty + 8 * k];
  }
}

}  // namespace

cudaError_t launch_fwd8(const Fwd8Args& a, bool causal, cudaStream_t st) {
  auto kern = causal ? fwd8_kernel<true> : fwd8_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int n_qblk = (a.N + NT * BM - 1) / (NT * BM);
  const long long grid = static_cast<long long>(n_qblk) * a.BH;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  trace_begin(TR_FWD8, st);
  kern<<<static_cast<unsigned>(grid), THREADS, SMEM_BYTES, st>>>(
      a.tmQ, a.tmK, a.tmVt, static_cast<__nv_bfloat16*>(a.O), a.L, a.N, n_qblk, a.group,
      a.c_log2, a.o_scale, a.ctl);
  e = cudaGetLastError();
  trace_end(TR_FWD8, st);
  return e;
}

cudaError_t launch_quant8(const void* X, void* Y, long long mats, int rows, int cols,
                          float inv_scale, bool transpose, bool bf16, cudaStream_t st) {
  const uint16_t* x = static_cast<const uint16_t*>(X);
  uint8_t* y = static_cast<uint8_t*>(Y);
  if (!transpose) {
    const long long n = mats * rows * cols;
    const long long blocks = std::min<long long>((n + 255) / 256, 152LL * 16);
    if (bf16)
      quant8_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, st>>>(x, y, n, inv_scale);
    else
      quant8_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, st>>>(x, y, n, inv_scale);
    return cudaGetLastError();
  }
  const dim3 grid((cols + 31) / 32, (rows + 31) / 32, static_cast<unsigned>(mats));
  const dim3 block(32, 8);
  if (bf16)
    quant8_t_kernel<true><<<grid, block, 0, st>>>(x, y, rows, cols, inv_scale);
  else
    quant8_t_kernel<false><<<grid, block, 0, st>>>(x, y, rows, cols, inv_scale);
  return cudaGetLastError();
}

}  // namespace fa
