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
// This file holds the pre-pass and the backward's entry:
//   pre_kernel   D = rowsum(dO o O) and L * log2(e), both laid out per 128-row
//                query block and padded (L -> +inf, D -> 0 past N) so the
//                dK/dV and dQ kernels (fa_bwd128.cu, every head dim) read them
//                with aligned loads.
#include "fa_internal.h"
#include "fa_ptx.cuh"

#include <type_traits>

namespace fa {

namespace {

constexpr int BM = 128;   // query rows per block (the padding unit of D and L)
constexpr float LOG2E = 1.4426950408889634f;

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
  grid_dep_launch();
  grid_dep_wait();             // O and L come from the forward
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
    cudaError_t e = launch_dependent(pre_kernel<D, BF16>, static_cast<unsigned>(blocks), 256, 0,
                                     st, a.O, a.dO, a.L, a.Dvec, Lp, a.N, Np, rows_p,
                                     a.cu_seqlens, a.H, a.total);
    trace_end(TR_BWD_PRE, st);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // dK/dV and dQ: the persistent kernels of fa_bwd64.cu at d <= 64, else fa_bwd128.cu's
  cudaError_t e = D <= 64 ? launch_dkdv64(a, D, BF16, CAUSAL, st)
                          : launch_dkdv128(a, D, BF16, CAUSAL, st);
  if (e != cudaSuccess) return e;
  return D <= 64 ? launch_dq64(a, D, BF16, CAUSAL, st) : launch_dq128(a, D, BF16, CAUSAL, st);
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
