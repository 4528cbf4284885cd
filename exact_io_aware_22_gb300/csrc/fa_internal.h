// fa_internal.h -- host-side interface between the C ABI (fa_api.cu) and the
// kernel launchers (fa_fwd.cu, fa_bwd.cu).  Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "fa_ptx.cuh"

namespace fa {

// Kernel kinds for the optional per-kernel CUDA-event trace (fa_trace_* in fa.h).
enum TraceKind {
  TR_FWD = 0,
  TR_BWD_PRE = 1,
  TR_BWD_DKDV = 2,
  TR_BWD_DQ = 3,
  TR_DEC_SPLIT = 4,
  TR_DEC_MERGE = 5,
  TR_FWD8 = 6,
  TR_NKINDS = 7
};
// Record an event before / after one kernel launch on `st` (no-op unless tracing).
void trace_begin(int kind, cudaStream_t st);
void trace_end(int kind, cudaStream_t st);

// Launch `kern` with programmatic stream serialisation: its CTAs may be scheduled
// while the previous kernel in `st` finishes its last wave, so launch latency and the
// kernel's set-up overlap that kernel's tail.  The kernel must call grid_dep_wait()
// before its first access to global memory that earlier work in the stream writes or
// reads (fa_ptx.cuh).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(KArgs...), unsigned grid, unsigned block,
                                    size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Heads per ordering group (block_pos) of a persistent kernel whose work items stream
// `bytes_per_head` bytes of one head's tiles: all heads (the whole grid longest-first)
// when they fit in about half of L2 together, else as many as do, at least 8.
inline int order_group(long long heads, long long bytes_per_head) {
  const long long budget = 64ll << 20;
  long long g = bytes_per_head > 0 ? budget / bytes_per_head : heads;
  if (g < 8) g = 8;
  if (g > heads) g = heads;
  return static_cast<int>(g < 1 ? 1 : g);
}

// Raise a kernel's dynamic shared-memory limit to `bytes`, once per kernel (later
// calls only look it up; launches from several host threads share the record).
inline cudaError_t ensure_smem(const void* kern, int bytes) {
  static std::mutex mu;
  static const void* seen[512];
  static int n_seen = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_seen; ++i)
    if (seen[i] == kern) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && n_seen < 512) seen[n_seen++] = kern;
  return e;
}

// TMA box of one 128-row tile: box_cols elements (one swizzle width) per row.
struct FwdTileInfo {
  int box_cols;
  int box_rows;
  int swizzle_bytes;
};
FwdTileInfo fwd_tile_info(int d);

struct FwdArgs {
  CUtensorMap tmQ, tmK, tmV;   // 3-D maps (d, N, B*H) of Q; (d, N, B*Hkv) of K and V
  void* O;
  float* L;
  int N, BH;
  int group;                   // query heads per K/V head (H / Hkv; 1 without sharing)
  int window;                  // causal sliding window of this many keys (0: none)
  // packed variable-length sequences (NULL: dense (B, H, N, d)): device int32
  // offsets [B+1]; Q, O (total, H, d), K, V (total, H/group, d), L (H, total); N is
  // then the longest sequence
  const int* cu_seqlens;
  int H, total;
  float c_log2;                // scale * log2(e)
  KernelCtl ctl;
};
cudaError_t launch_fwd(const FwdArgs& a, int d, bool bf16, bool causal, cudaStream_t st);

struct BwdArgs {
  CUtensorMap tmQ, tmK, tmV, tmO, tmdO;
  const void* Q;
  const void* O;
  const void* dO;
  const float* L;
  float* Dvec;                 // workspace: rowsum(dO o O), (B*H, N) fp32
  void* dQ;
  void* dK;
  void* dV;
  int N, BH;                   // BH = B*H query heads
  int group;                   // query heads per K/V head; B*H/group K/V heads
  int window;                  // causal sliding window of this many keys (0: none)
  const int* cu_seqlens;       // packed variable-length sequences, as in FwdArgs
  int H, total;
  float scale, c_log2;
  KernelCtl ctl;
};
cudaError_t launch_bwd(const BwdArgs& a, int d, bool bf16, bool causal, cudaStream_t st);
// dK/dV and dQ kernels after the pre-pass: the TMEM-resident kernels of fa_bwd128.cu
// (every head dim) and the persistent ones of fa_bwd64.cu (head dims 32 and 64)
cudaError_t launch_dkdv128(const BwdArgs& a, int d, bool bf16, bool causal, cudaStream_t st);
cudaError_t launch_dq128(const BwdArgs& a, int d, bool bf16, bool causal, cudaStream_t st);
cudaError_t launch_dkdv64(const BwdArgs& a, int d, bool bf16, bool causal, cudaStream_t st);
cudaError_t launch_dq64(const BwdArgs& a, int d, bool bf16, bool causal, cudaStream_t st);
// Workspace: D and L*log2(e) per padded row.
size_t bwd_workspace_bytes(long long BH, int N, int d);

struct DecodeArgs {
  CUtensorMap tmK, tmV;        // 3-D maps (d, Nmax, B*Hkv) of the caches, box decode_key_rows(d) rows
  const void* Q;               // (B, H, d) one query row per head
  const int* seqlens;          // device int32 [B]: cached keys per sequence
  void* O;                     // (B, H, d)
  float* L;                    // (B, H) fp32, natural log
  float* part;                 // workspace: (B*H, n_splits, d+4) partial states
  int B, H, Hkv, Nmax;
  int n_splits, chunk;         // splits of the cache and keys per split
  float c_log2;                // scale * log2(e) (E4M3 caches: times k_scale)
  float o_scale;               // 1 (E4M3 caches: v_scale)
  KernelCtl ctl;
};
// Query rows that one decode CTA serves from each K/V row (a power of two dividing H/Hkv).
int decode_rows(int H, int Hkv);
// Keys per ring stage of the decode kernel (the TMA box height); c8: E4M3 caches.
int decode_key_rows(int d, bool c8);
// Splits and keys per split (written to *chunk) for caches of Nmax keys.
int decode_parts(int B, int H, int Hkv, int Nmax, int* chunk);
cudaError_t launch_decode(const DecodeArgs& a, int d, bool bf16, bool c8, cudaStream_t st);

// Forward on 8-bit E4M3 inputs, d = 128, dense (B, H, N, 128) layout.
struct Fwd8Args {
  CUtensorMap tmQ, tmK;        // 3-D byte maps (128, N, B*H) / (128, N, B*Hkv), box 128 x 128
  CUtensorMap tmVt;            // 3-D byte map (N, 128, B*Hkv) of V^T, box 128 x 128
  void* O;                     // (B, H, N, 128) bf16
  float* L;                    // (B, H, N) fp32
  int N, BH, group;
  float c_log2;                // scale * q_scale * k_scale * log2(e)
  float o_scale;               // v_scale
  KernelCtl ctl;
};
cudaError_t launch_fwd8(const Fwd8Args& a, bool causal, cudaStream_t st);
// E4M3 codes of x * inv_scale for `mats` row-major rows x cols matrices of 16-bit
// values, optionally transposing each matrix.
cudaError_t launch_quant8(const void* X, void* Y, long long mats, int rows, int cols,
                          float inv_scale, bool transpose, bool bf16, cudaStream_t st);

}  // namespace fa
