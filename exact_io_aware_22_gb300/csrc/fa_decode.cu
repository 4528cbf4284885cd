// fa_decode.cu -- split-KV decoding: one new query row per (batch, head) against a
// key/value cache, on the CUDA cores.  Every cached K and V row is read once and
// serves all query rows that share its head, so the work is one read of the
// cache: HBM-bound, and a handful of query rows is far too narrow for tensor-core
// tiles.
//
// Method: the tutorial page "What is FlashAttention?", "Softmax in pieces": the
// softmax over disjoint key ranges is carried as partial states (m, l, acc) that
// merge exactly (m' = max(m1, m2), l' = l1 e^(m1-m') + l2 e^(m2-m'), acc likewise);
// inside one range, the running update of the docs page ("Tiling softmax is exact
// algebra", Fig. 3), in base 2 with scale * log2(e) folded into q.
//
//   decode_split_kernel  CTA = (batch, K/V head, group of R query heads, split of
//                        the cache); its four warps take consecutive quarters of the
//                        split.  Each warp streams its keys through its own two-stage
//                        ring of TMA tiles (KEYS keys of K and of V per stage, in the
//                        TMA swizzle, so that both access patterns below are free of
//                        bank conflicts) and keeps its own partial state:
//                          scores  lane = (column half, key): full dot products of
//                                  the R query rows (fp32, from shared memory) with
//                                  the lane's key, the halves summed by one shuffle;
//                          update  row maxima over the stage by shuffles, the
//                                  rescale factor and the probabilities, P written
//                                  to shared memory;
//                          P V     lane = D/32 output columns of all R rows, one
//                                  broadcast read of the stage's P row per key.
//                        The warps' states are merged in shared memory and written
//                        to the workspace, one (m, l, acc) record per row and split.
//   decode_merge_kernel  CTA = (batch, head): merges the records of the splits that
//                        hold keys; O = acc / l, L = (m + log2 l) ln 2.
#include "fa_internal.h"
#include "fa_ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace fa {

namespace {

constexpr int DEC_WARPS = 4;
constexpr int DEC_STAGES = 2;

// Geometry of one ring stage for head dim D, with 16-bit caches or (C8) E4M3 ones.
template <int D, bool C8 = false>
struct DecGeom {
  static constexpr int ELEM = C8 ? 1 : 2;              // bytes per cached value
  static constexpr int BOXC = C8 ? D : (D == 32 ? 32 : 64);   // columns of one TMA box
  static constexpr int ROWB = BOXC * ELEM;             // bytes of one box row (one swizzle span)
  static constexpr int SWM = ROWB == 128 ? 7 : 3;      // 16-byte chunk bits ^= row bits (128/64 B)
  static constexpr int HALVES = D / BOXC;              // lanes sharing one key in the score step
  static constexpr int KEYS = 32 / HALVES;             // keys per stage
  static constexpr int BOXB = KEYS * ROWB;             // bytes of one box (a multiple of 1 KiB)
  static constexpr int TILEB = HALVES * BOXB;          // K (or V) rows of one stage
  static constexpr int STAGEB = 2 * TILEB;             // K then V
  static constexpr int QS = HALVES * (BOXC + 4);       // floats per q row (halves 16 B apart mod 128)
  static constexpr int VEC = D / 32;                   // output columns per lane
};

template <int D, int R, bool C8>
constexpr int dec_smem_bytes() {
  using G = DecGeom<D, C8>;
  return 1024 + DEC_WARPS * DEC_STAGES * G::STAGEB + R * G::QS * 4 + DEC_WARPS * G::KEYS * R * 4 +
         DEC_WARPS * DEC_STAGES * 8;
}

// Byte offset of logical offset `off` inside a box laid out by the TMA swizzle
// (the 16-byte chunk index is XORed with the row bits above 128 bytes).
template <int SWM>
__device__ __forceinline__ uint32_t swz(uint32_t off) {
  return off ^ (((off >> 7) & SWM) << 4);
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a));
  return v;
}

// VEC 16-bit values at shared address a as floats.
template <int VEC, bool BF16>
__device__ __forceinline__ void lds_vec(uint32_t a, float (&out)[VEC]) {
  if constexpr (VEC == 4) {
    uint32_t x, y;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(x), "=r"(y) : "r"(a));
    const float2 p = unpack2<BF16>(x), q = unpack2<BF16>(y);
    out[0] = p.x; out[1] = p.y; out[2] = q.x; out[3] = q.y;
  } else if constexpr (VEC == 2) {
    uint32_t x;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(x) : "r"(a));
    const float2 p = unpack2<BF16>(x);
    out[0] = p.x; out[1] = p.y;
  } else {
    uint16_t x;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(x) : "r"(a));
    out[0] = unpack2<BF16>(static_cast<uint32_t>(x)).x;
  }
}

template <bool BF16>
__device__ __forceinline__ float load_f(const void* p, size_t i) {
  const uint16_t x = __ldg(static_cast<const uint16_t*>(p) + i);
  return unpack2<BF16>(static_cast<uint32_t>(x)).x;
}

// Four E4M3 codes (a 32-bit word) as floats.
__device__ __forceinline__ void e4m3x4_to_f(uint32_t w, float* out) {
  const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xffffu),
                                                     __NV_E4M3);
  const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16),
                                                     __NV_E4M3);
  const float2 a = __half22float2(__half2(lo)), b = __half22float2(__half2(hi));
  out[0] = a.x; out[1] = a.y; out[2] = b.x; out[3] = b.y;
}

template <int D, bool BF16, int R, bool C8>
__global__ void __launch_bounds__(32 * DEC_WARPS, 3)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const void* __restrict__ Q,
                        const int* __restrict__ seqlens, float* __restrict__ part, int H, int Hkv,
                        int Nmax, int chunk, int n_splits, float c_log2, KernelCtl ctl) {
  using G = DecGeom<D, C8>;
  constexpr int KEYS = G::KEYS, VEC = G::VEC;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_rc = (H / Hkv) / R;               // row groups per K/V head
  long long t = blockIdx.x;
  const int rc = static_cast<int>(t % n_rc);
  t /= n_rc;
  const int split = static_cast<int>(t % n_splits);
  const int bkv = static_cast<int>(t / n_splits);           // b * Hkv + hk
  const int b = bkv / Hkv, hk = bkv % Hkv;
  const int n = min(max(__ldg(seqlens + b), 0), Nmax);       // cached keys of this sequence
  const int s0 = split * chunk;
  if (s0 >= n) return;                          // no keys here; the merge skips this split
  const int s1 = min(s0 + chunk, n);
  // this warp's keys: whole stages, the last warp takes the remainder
  const int per = ((s1 - s0 + DEC_WARPS * KEYS - 1) / (DEC_WARPS * KEYS)) * KEYS;
  const int j0 = min(s0 + warp * per, s1), j1 = min(j0 + per, s1);
  const int nch = (j1 - j0 + KEYS - 1) / KEYS;
  const int h0 = (hk * (H / Hkv)) + rc * R;      // first query head of the group

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  const uint32_t ring = sb + warp * DEC_STAGES * G::STAGEB;
  const uint32_t qs = sb + DEC_WARPS * DEC_STAGES * G::STAGEB;
  const uint32_t ps = qs + R * G::QS * 4 + warp * KEYS * R * 4;
  const uint32_t bars = qs + R * G::QS * 4 + DEC_WARPS * KEYS * R * 4 + warp * DEC_STAGES * 8;
  float* qf = reinterpret_cast<float*>(smem_raw + (qs - raw));

  if (lane == 0) {
    for (int st = 0; st < DEC_STAGES; ++st) mbar_init(bars + st * 8, 1);
    fence_mbar_init();
  }
  // q * scale * log2(e) in fp32, the two column halves of a row 16 bytes apart mod 128
  for (int i = threadIdx.x; i < R * D; i += 32 * DEC_WARPS) {
    const int r = i / D, col = i % D;
    qf[r * G::QS + (col / G::BOXC) * (G::BOXC + 4) + col % G::BOXC] =
        load_f<BF16>(Q, (static_cast<size_t>(b) * H + h0 + r) * D + col) * c_log2;
  }
  __syncthreads();

  auto issue = [&](int c, int st) {
    const uint32_t bar = bars + st * 8, dst = ring + st * G::STAGEB;
    mbar_arrive_expect_tx(bar, G::STAGEB);
    const int y = j0 + c * KEYS;
#pragma unroll
    for (int bx = 0; bx < G::HALVES; ++bx) {
      tma_load_3d(dst + bx * G::BOXB, &tmK, bar, bx * G::BOXC, y, bkv);
      tma_load_3d(dst + G::TILEB + bx * G::BOXB, &tmV, bar, bx * G::BOXC, y, bkv);
    }
  };
  if (lane == 0)
    for (int c = 0; c < DEC_STAGES && c < nch; ++c) issue(c, c);

  const int key = lane % KEYS, half = lane / KEYS;
  float m[R], l[R], acc[R][VEC];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[r][e] = 0.f;
  }
  // shared offsets that do not change with the stage
  const uint32_t q_lane = qs + half * (G::BOXC + 4) * 4;
  const int col0 = lane * VEC;
  const uint32_t v_lane = (col0 / G::BOXC) * G::BOXB;
  const uint32_t v_col = (col0 % G::BOXC) * G::ELEM;

  int c = 0;
  for (; c < nch; ++c) {
    const int st = c % DEC_STAGES;
    if (!mbar_wait_warp(bars + st * 8, (c / DEC_STAGES) & 1, ctl)) break;
    const uint32_t kt = ring + st * G::STAGEB, vt = kt + G::TILEB;
    const int nk = min(KEYS, j1 - j0 - c * KEYS);

    // scores of the R rows with this lane's key over this lane's column half
    float2 s2[R];
#pragma unroll
    for (int r = 0; r < R; ++r) s2[r] = make_float2(0.f, 0.f);
    const uint32_t krow = kt + half * G::BOXB;
    if constexpr (C8) {
      // 16 E4M3 codes per 16-byte chunk of this lane's key row
#pragma unroll
      for (int cc = 0; cc < G::ROWB / 16; ++cc) {
        const uint4 kw = lds128(krow + swz<G::SWM>(key * G::ROWB + cc * 16));
        float k[16];
        e4m3x4_to_f(kw.x, k);
        e4m3x4_to_f(kw.y, k + 4);
        e4m3x4_to_f(kw.z, k + 8);
        e4m3x4_to_f(kw.w, k + 12);
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const float4 qv = lds128f(q_lane + (r * G::QS + cc * 16 + 4 * qq) * 4);
            s2[r] = fma2(make_float2(qv.x, qv.y), make_float2(k[4 * qq], k[4 * qq + 1]), s2[r]);
            s2[r] = fma2(make_float2(qv.z, qv.w), make_float2(k[4 * qq + 2], k[4 * qq + 3]), s2[r]);
          }
        }
      }
    } else {
#pragma unroll
      for (int cc = 0; cc < G::BOXC / 8; ++cc) {
        const uint4 kw = lds128(krow + swz<G::SWM>(key * G::ROWB + cc * 16));
        const float2 k0 = unpack2<BF16>(kw.x), k1 = unpack2<BF16>(kw.y);
        const float2 k2 = unpack2<BF16>(kw.z), k3 = unpack2<BF16>(kw.w);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float4 qa = lds128f(q_lane + (r * G::QS + cc * 8) * 4);
          const float4 qb = lds128f(q_lane + (r * G::QS + cc * 8 + 4) * 4);
          s2[r] = fma2(make_float2(qa.x, qa.y), k0, s2[r]);
          s2[r] = fma2(make_float2(qa.z, qa.w), k1, s2[r]);
          s2[r] = fma2(make_float2(qb.x, qb.y), k2, s2[r]);
          s2[r] = fma2(make_float2(qb.z, qb.w), k3, s2[r]);
        }
      }
    }
    const bool valid = key < nk;
    float p[R], alpha[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float s = s2[r].x + s2[r].y;
      if constexpr (G::HALVES == 2) s += __shfl_xor_sync(0xffffffffu, s, 16);
      s = valid ? s : -INFINITY;
      float mx = s;
#pragma unroll
      for (int w = KEYS / 2; w >= 1; w /= 2) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, w));
      const float m_new = fmaxf(m[r], mx);        // finite: the stage holds a key
      alpha[r] = ex2(m[r] - m_new);               // 0 at the first stage
      p[r] = ex2(s - m_new);                      // 0 for the masked lanes
      l[r] = fmaf(l[r], alpha[r], p[r]);          // this lane's key slot; summed at the end
      m[r] = m_new;
    }
    if (half == 0) {
      const uint32_t pa = ps + key * R * 4;
      if constexpr (R >= 4) {
#pragma unroll
        for (int r = 0; r < R; r += 4)
          asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(pa + r * 4), "f"(p[r]),
                       "f"(p[r + 1]), "f"(p[r + 2]), "f"(p[r + 3])
                       : "memory");
      } else {
#pragma unroll
        for (int r = 0; r < R; ++r)
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(pa + r * 4), "f"(p[r]) : "memory");
      }
    }
    __syncwarp();
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[r][e] *= alpha[r];
#pragma unroll 4
    for (int kk = 0; kk < nk; ++kk) {
      float pv[R];
      if constexpr (R >= 4) {
#pragma unroll
        for (int r = 0; r < R; r += 4) {
          const float4 t4 = lds128f(ps + (kk * R + r) * 4);
          pv[r] = t4.x; pv[r + 1] = t4.y; pv[r + 2] = t4.z; pv[r + 3] = t4.w;
        }
      } else {
#pragma unroll
        for (int r = 0; r < R; ++r)
          asm volatile("ld.shared.f32 %0, [%1];" : "=f"(pv[r]) : "r"(ps + (kk * R + r) * 4));
      }
      float v[VEC];
      if constexpr (C8) {                        // VEC = 4 codes, one 32-bit word
        uint32_t x;
        asm volatile("ld.shared.b32 %0, [%1];"
                     : "=r"(x)
                     : "r"(vt + v_lane + swz<G::SWM>(kk * G::ROWB + v_col)));
        e4m3x4_to_f(x, v);
      } else {
        lds_vec<VEC, BF16>(vt + v_lane + swz<G::SWM>(kk * G::ROWB + v_col), v);
      }
      if constexpr (VEC % 2 == 0) {               // pairs of columns: packed fp32x2 FMAs
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float2 p2 = make_float2(pv[r], pv[r]);
#pragma unroll
          for (int e = 0; e < VEC; e += 2) {
            const float2 a = fma2(p2, make_float2(v[e], v[e + 1]), make_float2(acc[r][e], acc[r][e + 1]));
            acc[r][e] = a.x;
            acc[r][e + 1] = a.y;
          }
        }
      } else {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[r][e] = fmaf(pv[r], v[e], acc[r][e]);
      }
    }
    __syncwarp();                                 // stage and P read by every lane
    if (lane == 0 && c + DEC_STAGES < nch) issue(c + DEC_STAGES, st);
  }
  if (c < nch) {
    // a wait ran out (recorded in the status word): let the copies already issued
    // land (bounded) before the CTA's shared memory is released
    for (int k = c; k < nch && k < c + DEC_STAGES; ++k)
      mbar_wait_warp(bars + (k % DEC_STAGES) * 8, (k / DEC_STAGES) & 1, ctl);
  }

  // the four warps' states merged into one per row (the merge of two partial states,
  // applied across the warps), staged in the ring's shared memory once every warp is
  // done with its ring; then one (m, l, -, -, acc[D]) record per row and split
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int w = KEYS / 2; w >= 1; w /= 2) l[r] += __shfl_xor_sync(0xffffffffu, l[r], w);
  __syncthreads();
  float* red = reinterpret_cast<float*>(smem_raw + (sb - raw));   // [W][R] (m, l), [W][R][D] acc
  float* racc = red + 2 * DEC_WARPS * R;
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      red[(warp * R + r) * 2] = m[r];
      red[(warp * R + r) * 2 + 1] = l[r];
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int e = 0; e < VEC; ++e) racc[(warp * R + r) * D + col0 + e] = acc[r][e];
  __syncthreads();
  for (int i = threadIdx.x; i < R * D; i += 32 * DEC_WARPS) {
    const int r = i / D, col = i % D;
    float mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < DEC_WARPS; ++w) mm = fmaxf(mm, red[(w * R + r) * 2]);   // finite: warp 0 has keys
    float ll = 0.f, aa = 0.f;
#pragma unroll
    for (int w = 0; w < DEC_WARPS; ++w) {
      const float a = ex2(red[(w * R + r) * 2] - mm);   // an empty warp (m = -inf) weighs 0
      ll = fmaf(red[(w * R + r) * 2 + 1], a, ll);
      aa = fmaf(racc[(w * R + r) * D + col], a, aa);
    }
    float* dst = part + ((static_cast<size_t>(b) * H + h0 + r) * n_splits + split) * (D + 4);
    dst[4 + col] = aa;
    if (col == 0) {
      dst[0] = mm;
      dst[1] = ll;
    }
  }
}

// ---------------------------------------------------------------- E4M3 caches
// The split kernel for E4M3 caches (d = 128) forms scores and P.V with warp-level
// tensor-core products (mma.sync m16n8k16, f16 operands, fp32 accumulation) instead
// of per-key FMAs, so each key costs a code conversion and a share of 64 MMAs per
// 32-key stage rather than 2 x 128 FMAs per query row: the cache read, not the issue
// slots, then sets the pace.  E4M3 codes convert to f16 exactly (cvt of two codes per
// instruction); q is taken as f16 (exact for fp16 input, and for bf16 values inside
// f16's range) and the scale is applied to the fp32 scores; P is rounded to f16 for
// the P.V product (the row sums use the fp32 values).
//   rows     query row g = lane / 4 of the group (rows >= R are zero padding)
//   scores   the head dim is visited in an order of its own, the same for q and K:
//            k-step ks, fragment column 2c + e (e = 0, 1) and 2c + 8 + e stand for
//            dims 32c + 4ks + e and 32c + 4ks + 2 + e (c = lane % 4), so lane (g, c)
//            reads 32 contiguous bytes of its key row per 8-key tile.
//   P.V      the score fragments of two key tiles are the A fragment of one 16-key
//            k-step (P never leaves registers); output fragment column n of tile jn
//            stands for dim 16n + jn, so lane (g, c) reads 16 contiguous bytes of each
//            of its four V rows, and holds dims 32c + jn and 32c + 16 + jn.
__device__ __forceinline__ uint32_t cvt_e4m3x2_f16x2(uint32_t codes16) {
  uint32_t r;
  asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}"
      : "=r"(r)
      : "r"(codes16));
  return r;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a2, uint32_t b0,
                                         uint32_t b1) {
  // rows g + 8 of A are zero (a1 = a3 = 0)
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t f2_to_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <bool BF16, int R>
__global__ void __launch_bounds__(32 * DEC_WARPS, 3)
    decode8_split_kernel(const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const void* __restrict__ Q,
                         const int* __restrict__ seqlens, float* __restrict__ part, int H, int Hkv,
                         int Nmax, int chunk, int n_splits, float c_log2, KernelCtl ctl) {
  constexpr int D = 128;
  using G = DecGeom<D, true>;
  constexpr int KEYS = G::KEYS;                 // 32 keys per stage, one 128-byte row each
  static_assert(KEYS == 32 && G::ROWB == 128 && G::HALVES == 1, "E4M3 stage geometry");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, cq = lane & 3;      // fragment row, column pair
  const int n_rc = (H / Hkv) / R;               // row groups per K/V head
  long long t = blockIdx.x;
  const int rc = static_cast<int>(t % n_rc);
  t /= n_rc;
  const int split = static_cast<int>(t % n_splits);
  const int bkv = static_cast<int>(t / n_splits);           // b * Hkv + hk
  const int b = bkv / Hkv, hk = bkv % Hkv;
  const int n = min(max(__ldg(seqlens + b), 0), Nmax);       // cached keys of this sequence
  const int s0 = split * chunk;
  if (s0 >= n) return;                          // no keys here; the merge skips this split
  const int s1 = min(s0 + chunk, n);
  const int per = ((s1 - s0 + DEC_WARPS * KEYS - 1) / (DEC_WARPS * KEYS)) * KEYS;
  const int j0 = min(s0 + warp * per, s1), j1 = min(j0 + per, s1);
  const int nch = (j1 - j0 + KEYS - 1) / KEYS;
  const int h0 = (hk * (H / Hkv)) + rc * R;      // first query head of the group

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  const uint32_t ring = sb + warp * DEC_STAGES * G::STAGEB;
  const uint32_t bars = sb + DEC_WARPS * DEC_STAGES * G::STAGEB + warp * DEC_STAGES * 8;
  if (lane == 0) {
    for (int st = 0; st < DEC_STAGES; ++st) mbar_init(bars + st * 8, 1);
    fence_mbar_init();
  }
  // q of row gq as the A fragments of the score products, in f16 (rows >= R: zero)
  uint32_t qa[8][2];
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (gq < R) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        v[e] = load_f<BF16>(Q, (static_cast<size_t>(b) * H + h0 + gq) * D + 32 * cq + 4 * ks + e);
    }
    qa[ks][0] = f2_to_h2(v[0], v[1]);
    qa[ks][1] = f2_to_h2(v[2], v[3]);
  }
  __syncwarp();

  auto issue = [&](int c, int st) {
    const uint32_t bar = bars + st * 8, dst = ring + st * G::STAGEB;
    mbar_arrive_expect_tx(bar, G::STAGEB);
    const int y = j0 + c * KEYS;
    tma_load_3d(dst, &tmK, bar, 0, y, bkv);
    tma_load_3d(dst + G::TILEB, &tmV, bar, 0, y, bkv);
  };
  if (lane == 0)
    for (int c = 0; c < DEC_STAGES && c < nch; ++c) issue(c, c);

  float m_row = -INFINITY, l_part = 0.f;        // row gq: running max, this lane's part of l
  float acc[16][4];                             // P.V fragments of 16 output tiles
#pragma unroll
  for (int jn = 0; jn < 16; ++jn)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[jn][e] = 0.f;

  int c = 0;
  for (; c < nch; ++c) {
    const int st = c % DEC_STAGES;
    if (!mbar_wait_warp(bars + st * 8, (c / DEC_STAGES) & 1, ctl)) break;
    const uint32_t kt = ring + st * G::STAGEB, vt = kt + G::TILEB;
    const int nk = min(KEYS, j1 - j0 - c * KEYS);

    // scores of row gq with keys 8j + 2cq + e (e = 0, 1), j = 0..3
    float s[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[j][e] = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int key = 8 * j + gq;
      const uint4 wa = lds128(kt + swz<G::SWM>(key * G::ROWB + 32 * cq));
      const uint4 wb = lds128(kt + swz<G::SWM>(key * G::ROWB + 32 * cq + 16));
      const uint32_t w[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma16816(s[j], qa[ks][0], qa[ks][1], cvt_e4m3x2_f16x2(w[ks] & 0xffffu),
                 cvt_e4m3x2_f16x2(w[ks] >> 16));
    }
    // online update of row gq over this stage's keys (keys past nk: -inf)
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = 8 * j + 2 * cq + e;
        s[j][e] = key < nk ? s[j][e] * c_log2 : -INFINITY;
        mx = fmaxf(mx, s[j][e]);
      }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m_row, mx);       // finite: the stage holds a key
    const float alpha = ex2(m_row - m_new);     // 0 at the first stage
    m_row = m_new;
    float p[4][2];
    float ps = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        p[j][e] = ex2(s[j][e] - m_new);         // 0 for keys past nk
        ps += p[j][e];
      }
    l_part = fmaf(l_part, alpha, ps);
#pragma unroll
    for (int jn = 0; jn < 16; ++jn) {
      acc[jn][0] *= alpha;
      acc[jn][1] *= alpha;
    }
    // P.V: k-step kk covers keys 16kk .. 16kk + 15; V rows past nk read as zero
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const uint32_t pa0 = f2_to_h2(p[2 * kk][0], p[2 * kk][1]);
      const uint32_t pa2 = f2_to_h2(p[2 * kk + 1][0], p[2 * kk + 1][1]);
      const int r0 = 16 * kk + 2 * cq;          // rows r0, r0 + 1 (b0) and r0 + 8, r0 + 9 (b1)
      uint4 v4[4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int vr = r0 + (q4 & 1) + 8 * (q4 >> 1);
        v4[q4] = lds128(vt + swz<G::SWM>(vr * G::ROWB + 16 * gq));
        if (vr >= nk) v4[q4] = make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int wd = 0; wd < 4; ++wd) {
        const uint32_t A0 = (&v4[0].x)[wd], A1 = (&v4[1].x)[wd];   // rows r0, r0 + 1
        const uint32_t B0 = (&v4[2].x)[wd], B1 = (&v4[3].x)[wd];   // rows r0 + 8, r0 + 9
        const uint32_t lo0 = prmt(A0, A1, 0x5140u), hi0 = prmt(A0, A1, 0x7362u);
        const uint32_t lo1 = prmt(B0, B1, 0x5140u), hi1 = prmt(B0, B1, 0x7362u);
        mma16816(acc[4 * wd + 0], pa0, pa2, cvt_e4m3x2_f16x2(lo0 & 0xffffu), cvt_e4m3x2_f16x2(lo1 & 0xffffu));
        mma16816(acc[4 * wd + 1], pa0, pa2, cvt_e4m3x2_f16x2(lo0 >> 16), cvt_e4m3x2_f16x2(lo1 >> 16));
        mma16816(acc[4 * wd + 2], pa0, pa2, cvt_e4m3x2_f16x2(hi0 & 0xffffu), cvt_e4m3x2_f16x2(hi1 & 0xffffu));
        mma16816(acc[4 * wd + 3], pa0, pa2, cvt_e4m3x2_f16x2(hi0 >> 16), cvt_e4m3x2_f16x2(hi1 >> 16));
      }
    }
    __syncwarp();                                 // stage read by every lane
    if (lane == 0 && c + DEC_STAGES < nch) issue(c + DEC_STAGES, st);
  }
  if (c < nch) {
    // a wait ran out (recorded in the status word): let the copies already issued
    // land (bounded) before the CTA's shared memory is released
    for (int k = c; k < nch && k < c + DEC_STAGES; ++k)
      mbar_wait_warp(bars + (k % DEC_STAGES) * 8, (k / DEC_STAGES) & 1, ctl);
  }

  // row sums over the four lanes of a row; the warps' states merged per row in shared
  // memory (staged in the ring once every warp is done with it); one record per row and split
  l_part += __shfl_xor_sync(0xffffffffu, l_part, 1);
  l_part += __shfl_xor_sync(0xffffffffu, l_part, 2);
  __syncthreads();
  float* red = reinterpret_cast<float*>(smem_raw + (sb - raw));   // [W][R] (m, l), [W][R][D] acc
  float* racc = red + 2 * DEC_WARPS * R;
  if (gq < R) {
    if (cq == 0) {
      red[(warp * R + gq) * 2] = m_row;
      red[(warp * R + gq) * 2 + 1] = l_part;
    }
#pragma unroll
    for (int jn = 0; jn < 16; ++jn) {
      racc[(warp * R + gq) * D + 32 * cq + jn] = acc[jn][0];
      racc[(warp * R + gq) * D + 32 * cq + 16 + jn] = acc[jn][1];
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < R * D; i += 32 * DEC_WARPS) {
    const int r = i / D, col = i % D;
    float mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < DEC_WARPS; ++w) mm = fmaxf(mm, red[(w * R + r) * 2]);   // finite: warp 0 has keys
    float ll = 0.f, aa = 0.f;
#pragma unroll
    for (int w = 0; w < DEC_WARPS; ++w) {
      const float a = ex2(red[(w * R + r) * 2] - mm);   // an empty warp (m = -inf) weighs 0
      ll = fmaf(red[(w * R + r) * 2 + 1], a, ll);
      aa = fmaf(racc[(w * R + r) * D + col], a, aa);
    }
    float* dst = part + ((static_cast<size_t>(b) * H + h0 + r) * n_splits + split) * (D + 4);
    dst[4 + col] = aa;
    if (col == 0) {
      dst[0] = mm;
      dst[1] = ll;
    }
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(D)
    decode_merge_kernel(const float* __restrict__ part, const int* __restrict__ seqlens,
                        void* __restrict__ O, float* __restrict__ L, int H, int Nmax, int chunk,
                        int n_splits, float o_scale) {
  const size_t row = blockIdx.x;                 // b * H + h
  const int b = static_cast<int>(row / H);
  const int n = min(max(__ldg(seqlens + b), 0), Nmax);
  const int used = (n + chunk - 1) / chunk;      // splits that wrote a record for this row
  const float* src = part + row * n_splits * (D + 4);
  // launched as a programmatic dependent of the split kernel: wait for its results
  asm volatile("griddepcontrol.wait;" ::: "memory");
  float m = -INFINITY;
  for (int p = 0; p < used; ++p) m = fmaxf(m, src[p * (D + 4)]);
  float l = 0.f, acc = 0.f;
  if (m != -INFINITY) {                          // no key at all: l = 0, acc = 0
#pragma unroll 4
    for (int p = 0; p < used; ++p) {
      const float* sp = src + p * (D + 4);
      const float a = ex2(sp[0] - m);
      l = fmaf(sp[1], a, l);
      acc = fmaf(sp[4 + threadIdx.x], a, acc);
    }
  }
  const float o = l > 0.f ? acc / l * o_scale : 0.f;
  if constexpr (BF16)
    reinterpret_cast<__nv_bfloat16*>(O)[row * D + threadIdx.x] = __float2bfloat16_rn(o);
  else
    reinterpret_cast<__half*>(O)[row * D + threadIdx.x] = __float2half_rn(o);
  if (threadIdx.x == 0) L[row] = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
}

template <int D, bool BF16, int R, bool C8>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t st) {
  constexpr int smem = dec_smem_bytes<D, R, C8>();
  void (*kern)(const CUtensorMap, const CUtensorMap, const void*, const int*, float*, int, int,
               int, int, int, float, KernelCtl);
  if constexpr (C8) kern = decode8_split_kernel<BF16, R>;
  else kern = decode_split_kernel<D, BF16, R, C8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long ctas =
      static_cast<long long>(a.B) * a.Hkv * a.n_splits * ((a.H / a.Hkv) / R);
  trace_begin(TR_DEC_SPLIT, st);
  kern<<<static_cast<unsigned>(ctas), 32 * DEC_WARPS, smem, st>>>(
      a.tmK, a.tmV, a.Q, a.seqlens, a.part, a.H, a.Hkv, a.Nmax, a.chunk, a.n_splits, a.c_log2,
      a.ctl);
  e = cudaGetLastError();
  trace_end(TR_DEC_SPLIT, st);
  if (e != cudaSuccess) return e;
  // the merge may be scheduled while the split kernel drains; it waits for the
  // split kernel's writes (griddepcontrol.wait) before reading them
  trace_begin(TR_DEC_MERGE, st);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(static_cast<long long>(a.B) * a.H));
  cfg.blockDim = dim3(D);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_merge_kernel<D, BF16>, static_cast<const float*>(a.part),
                         a.seqlens, a.O, a.L, a.H, a.Nmax, a.chunk, a.n_splits, a.o_scale);
  trace_end(TR_DEC_MERGE, st);
  return e;
}

template <int D, bool BF16, bool C8 = false>
cudaError_t launch_decode_d(const DecodeArgs& a, cudaStream_t st) {
  switch (decode_rows(a.H, a.Hkv)) {
    case 8: return launch_decode_t<D, BF16, 8, C8>(a, st);
    case 4: return launch_decode_t<D, BF16, 4, C8>(a, st);
    case 2: return launch_decode_t<D, BF16, 2, C8>(a, st);
    default: return launch_decode_t<D, BF16, 1, C8>(a, st);
  }
}

}  // namespace

int decode_rows(int H, int Hkv) {
  const int g = H / Hkv;
  return g % 8 == 0 ? 8 : g % 4 == 0 ? 4 : g % 2 == 0 ? 2 : 1;
}

int decode_parts(int B, int H, int Hkv, int Nmax, int* chunk) {
  // about sixteen CTAs per SM (152 SMs; three are resident at a time, so the last
  // wave is short), each with at least 256 keys
  const long long groups = static_cast<long long>(B) * Hkv * ((H / Hkv) / decode_rows(H, Hkv));
  long long splits = (16 * 152 + groups - 1) / groups;
  const long long max_splits = (static_cast<long long>(Nmax) + 255) / 256;
  if (splits > max_splits) splits = max_splits;
  if (splits < 1) splits = 1;
  // keys per split: a multiple of 64, so every warp but the last takes whole stages
  long long c = (Nmax + splits - 1) / splits;
  c = (c + 63) / 64 * 64;
  *chunk = static_cast<int>(c);
  return static_cast<int>((Nmax + c - 1) / c);
}

int decode_key_rows(int d, bool c8) { return (d == 128 && !c8) ? 16 : 32; }

cudaError_t launch_decode(const DecodeArgs& a, int d, bool bf16, bool c8, cudaStream_t st) {
  if (c8) {                                      // E4M3 caches: d = 128
    if (d != 128) return cudaErrorInvalidValue;
    return bf16 ? launch_decode_d<128, true, true>(a, st) : launch_decode_d<128, false, true>(a, st);
  }
  if (d == 32) return bf16 ? launch_decode_d<32, true>(a, st) : launch_decode_d<32, false>(a, st);
  if (d == 64) return bf16 ? launch_decode_d<64, true>(a, st) : launch_decode_d<64, false>(a, st);
  if (d == 128)
    return bf16 ? launch_decode_d<128, true>(a, st) : launch_decode_d<128, false>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace fa
