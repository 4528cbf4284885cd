// fa_api.cu -- the C ABI declared in include/fa.h: argument validation,
// TMA tensor-map encoding, workspace handling, the device status word, and
// dispatch to the forward / backward launchers.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

// Sticky status word written by kernels whose bounded wait ran out.
__device__ uint32_t g_status_word;

unsigned long long g_wait_limit_ns = 2000000000ull;
thread_local int g_last_cuda_error = 0;

fa_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return FA_ERR_CUDA;
}

// ---- device addresses of this library's file-scope __device__ variables
// On the host a __device__ variable's name is only a stand-in; its device address
// belongs to one CUDA context (the module is loaded anew into every context, and a
// context that is destroyed and recreated, e.g. by cudaDeviceReset, may place it
// elsewhere).  Addresses are therefore cached per context, keyed on the driver's
// unique context ID (never reused within a process), and looked up again in a new
// context.  One lock guards the table, so first calls from several host threads do
// not race.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

fa_status driver_fn(const char* name, void** fn) {
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion(name, fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess) return cuda_fail(e);
  if (q != cudaDriverEntryPointSuccess || !*fn) return cuda_fail(cudaErrorSymbolNotFound);
  return FA_OK;
}

// ID of the context current on this thread (0: none yet).
fa_status current_ctx_id(unsigned long long* id) {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  static fa_status init_st = FA_OK;
  std::call_once(once, [] {
    void* a = nullptr;
    void* b = nullptr;
    init_st = driver_fn("cuCtxGetCurrent", &a);
    if (init_st == FA_OK) init_st = driver_fn("cuCtxGetId", &b);
    get_cur = reinterpret_cast<CtxGetCurrentFn>(a);
    get_id = reinterpret_cast<CtxGetIdFn>(b);
  });
  if (init_st != FA_OK) return init_st;
  CUcontext ctx = nullptr;
  if (get_cur(&ctx) != CUDA_SUCCESS) return cuda_fail(cudaErrorContextIsDestroyed);
  *id = 0;
  if (ctx && get_id(ctx, id) != CUDA_SUCCESS) return cuda_fail(cudaErrorContextIsDestroyed);
  return FA_OK;
}

// Device address of the __device__ variable `sym` in the current context.
fa_status symbol_address(const void* sym, void** out) {
  struct Entry {
    unsigned long long ctx;
    const void* sym;
    void* ptr;
  };
  constexpr int kEntries = 64;
  static Entry table[kEntries] = {};
  static int next = 0;
  static std::mutex mu;
  unsigned long long id = 0;
  fa_status st = current_ctx_id(&id);
  if (st != FA_OK) return st;
  std::lock_guard<std::mutex> lock(mu);
  if (id != 0)
    for (const Entry& en : table)
      if (en.ctx == id && en.sym == sym) {
        *out = en.ptr;
        return FA_OK;
      }
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, sym);   // also creates the context if needed
  if (e != cudaSuccess) return cuda_fail(e);
  if (id == 0 && (st = current_ctx_id(&id)) != FA_OK) return st;
  if (id != 0) {
    table[next] = {id, sym, p};
    next = (next + 1) % kEntries;
  }
  *out = p;
  return FA_OK;
}

// Device address of the status word in the current context.
fa_status status_ptr(uint32_t** out) {
  void* p = nullptr;
  fa_status st = symbol_address(reinterpret_cast<const void*>(&g_status_word), &p);
  if (st != FA_OK) return st;
  *out = static_cast<uint32_t*>(p);
  return FA_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

fa_status get_encoder(EncodeTiledFn* fn) {
  static EncodeTiledFn cached = nullptr;
  if (!cached) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess) return cuda_fail(e);
    if (q != cudaDriverEntryPointSuccess || !p) return cuda_fail(cudaErrorSymbolNotFound);
    cached = reinterpret_cast<EncodeTiledFn>(p);
  }
  *fn = cached;
  return FA_OK;
}

// 3-D map (d, N, B*H) over a dense (B,H,N,d) 16-bit array; box = one 128-row
// tile of one swizzle width.  Rows >= N of a head read as zeros.
fa_status make_map(CUtensorMap* m, const void* base, int d, int N, long long BH, bool bf16,
                   int box_rows = 128) {
  EncodeTiledFn enc;
  fa_status st = get_encoder(&enc);
  if (st != FA_OK) return st;
  fa::FwdTileInfo ti = fa::fwd_tile_info(d);
  ti.box_rows = box_rows;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(ti.box_cols), static_cast<cuuint32_t>(ti.box_rows),
                       1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   ti.swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return FA_OK;
}

// 3-D map (d, Hx, total) over packed sequences (total, Hx, d): box = one head of one
// 128-row tile of one swizzle width, laid out in shared memory as make_map's tile.
// Rows >= total read as zeros.
fa_status make_map_packed(CUtensorMap* m, const void* base, int d, int Hx, int total, bool bf16) {
  EncodeTiledFn enc;
  fa_status st = get_encoder(&enc);
  if (st != FA_OK) return st;
  const fa::FwdTileInfo ti = fa::fwd_tile_info(d);
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Hx),
                        static_cast<cuuint64_t>(total)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(Hx) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(ti.box_cols), 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   ti.swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return FA_OK;
}

// 3-D map over bytes (inner, rows, depth), box 128 bytes x box_rows x 1 in the
// 128-byte swizzle: the 8-bit tiles of the E4M3 forward and of E4M3 caches.  Elements
// past the edges read as 0.
fa_status make_map_bytes(CUtensorMap* m, const void* base, long long inner, long long rows,
                         long long depth, unsigned box_rows = 128) {
  EncodeTiledFn enc;
  fa_status st = get_encoder(&enc);
  if (st != FA_OK) return st;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(depth)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner),
                           static_cast<cuuint64_t>(inner) * static_cast<cuuint64_t>(rows)};
  cuuint32_t box[3] = {128, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return FA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Shared validation of sizes, dtype and scale.
fa_status check_common(int B, int H, int N, int d, int causal, float scale, int dtype) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_VALUE;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_VALUE;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_VALUE;
  if (d != 32 && d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * H;
  const long long nblk = (static_cast<long long>(N) + 127) / 128;
  if (BH > 0x7fffffffLL || nblk * BH > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(N) * d * 2 >= (1LL << 40)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

fa_status ctl_for_launch(fa::KernelCtl* ctl) {
  fa_status st = status_ptr(&ctl->status);
  if (st != FA_OK) return st;
  ctl->wait_limit_ns = g_wait_limit_ns;
  return FA_OK;
}

__global__ void selftest_wait_kernel(fa::KernelCtl ctl) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = fa::smem_u32(&bar);
  if (threadIdx.x == 0) {
    fa::mbar_init(b, 1);
    fa::fence_mbar_init();
    // nothing ever arrives: the bounded wait must give up and record it
    fa::mbar_wait(b, 0, ctl);
  }
}

// ---- per-kernel trace: a fixed pool of event pairs, filled in launch order
constexpr int kTracePool = 4096;
struct TraceRec {
  cudaEvent_t start, stop;
  int kind;
};
TraceRec g_trace[kTracePool];
bool g_trace_created = false;
bool g_trace_on = false;
int g_trace_n = 0;
int g_trace_open = -1;   // record whose stop event is pending

const char* const kTraceNames[fa::TR_NKINDS] = {"fwd_kernel",      "bwd_pre_kernel",
                                                 "bwd_dkdv_kernel", "bwd_dq_kernel",
                                                 "decode_split_kernel", "decode_merge_kernel",
                                                 "fwd_fp8_kernel"};

}  // namespace

namespace fa {
void trace_begin(int kind, cudaStream_t st) {
  if (!g_trace_on || g_trace_n >= kTracePool) return;
  TraceRec& r = g_trace[g_trace_n];
  if (cudaEventRecord(r.start, st) != cudaSuccess) return;
  r.kind = kind;
  g_trace_open = g_trace_n;
}
void trace_end(int kind, cudaStream_t st) {
  if (!g_trace_on || g_trace_open < 0) return;
  TraceRec& r = g_trace[g_trace_open];
  g_trace_open = -1;
  if (r.kind != kind || cudaEventRecord(r.stop, st) != cudaSuccess) return;
  ++g_trace_n;
}
}  // namespace fa

extern "C" {

fa_status fa_trace_enable(int on) {
  if (on) {
    if (!g_trace_created) {
      for (int i = 0; i < kTracePool; ++i) {
        cudaError_t e = cudaEventCreate(&g_trace[i].start);
        if (e == cudaSuccess) e = cudaEventCreate(&g_trace[i].stop);
        if (e != cudaSuccess) return cuda_fail(e);
      }
      g_trace_created = true;
    }
    g_trace_n = 0;
    g_trace_open = -1;
  }
  g_trace_on = on != 0;
  return FA_OK;
}

const char* fa_trace_kind_name(int kind) {
  return (kind >= 0 && kind < fa::TR_NKINDS) ? kTraceNames[kind] : nullptr;
}

fa_status fa_trace_read(int kind, double* total_ms, long long* launches) {
  if (!total_ms || !launches || kind < 0 || kind >= fa::TR_NKINDS) return FA_ERR_INVALID_VALUE;
  double t = 0.0;
  long long n = 0;
  for (int i = 0; i < g_trace_n; ++i) {
    if (g_trace[i].kind != kind) continue;
    cudaError_t e = cudaEventSynchronize(g_trace[i].stop);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, g_trace[i].start, g_trace[i].stop);
    if (e != cudaSuccess) return cuda_fail(e);
    t += ms;
    ++n;
  }
  *total_ms = t;
  *launches = n;
  return FA_OK;
}


const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_VALUE: return "FA_ERR_INVALID_VALUE: invalid argument";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: head dim, dtype or size not supported";
    case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED: pointer alignment rule violated";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: CUDA call or kernel launch failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel gave up a bounded wait";
  }
  return "unknown fa_status";
}

int fa_last_cuda_error(void) { return g_last_cuda_error; }

fa_status fa_set_wait_limit_ns(unsigned long long ns) {
  g_wait_limit_ns = ns ? ns : 2000000000ull;
  return FA_OK;
}

fa_status fa_device_status(void* stream) {
  uint32_t* p = nullptr;
  fa_status st = status_ptr(&p);
  if (st != FA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e);
  uint32_t v = 0;
  e = cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  const uint32_t zero = 0;
  e = cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e);
  if (v & fa::FA_DEV_TIMEOUT) return FA_ERR_TIMEOUT;
  return (v & fa::FA_DEV_SMEM_ALIGN) ? FA_ERR_UNSUPPORTED : FA_OK;
}

fa_status fa_selftest_timeout(unsigned long long limit_ns, void* stream) {
  fa::KernelCtl ctl;
  fa_status st = ctl_for_launch(&ctl);
  if (st != FA_OK) return st;
  ctl.wait_limit_ns = limit_ns ? limit_ns : 1000000ull;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(ctl);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return fa_device_status(stream);
}

// Hkv K/V heads shared by groups of H/Hkv consecutive query heads (Hkv == H: no sharing).
static fa_status check_heads(int H, int Hkv) {
  if (Hkv < 1 || Hkv > H || H % Hkv != 0) return FA_ERR_INVALID_VALUE;
  return FA_OK;
}

// Packed variable-length sequences (cu_seqlens != NULL): N is the longest sequence,
// `total` the packed row count; Q, O (total, H, d), K, V (total, Hkv, d), L (H, total).
static fa_status check_packed(const int* cu_seqlens, int total) {
  if (!cu_seqlens || total < 1) return FA_ERR_INVALID_VALUE;
  if (!aligned(cu_seqlens, 4)) return FA_ERR_MISALIGNED;
  return FA_OK;
}

static fa_status fwd_impl(const void* Q, const void* K, const void* V, void* O, float* L, int B,
                          int H, int Hkv, int N, int d, int causal, float scale, fa_dtype dtype,
                          void* stream, int window = 0, const int* cu_seqlens = nullptr,
                          int total = 0) {
  fa_status st = check_common(B, H, N, d, causal, scale, static_cast<int>(dtype));
  if (st != FA_OK) return st;
  if ((st = check_heads(H, Hkv)) != FA_OK) return st;
  if (cu_seqlens && (st = check_packed(cu_seqlens, total)) != FA_OK) return st;
  if (!Q || !K || !V || !O || !L) return FA_ERR_INVALID_VALUE;
  if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) || !aligned(L, 4))
    return FA_ERR_MISALIGNED;
  const long long BH = static_cast<long long>(B) * H, BHkv = static_cast<long long>(B) * Hkv;
  const size_t rows = cu_seqlens ? static_cast<size_t>(total) : static_cast<size_t>(B) * N;
  const size_t nbytes = rows * H * d * 2, lbytes = rows * H * 4;
  const size_t kvbytes = rows * Hkv * d * 2;
  const void* ins[3] = {Q, K, V};
  const size_t insz[3] = {nbytes, kvbytes, kvbytes};
  for (int i = 0; i < 3; ++i)
    if (overlap(ins[i], insz[i], O, nbytes) || overlap(ins[i], insz[i], L, lbytes))
      return FA_ERR_INVALID_VALUE;
  if (overlap(O, nbytes, L, lbytes)) return FA_ERR_INVALID_VALUE;

  const bool bf16 = dtype == FA_BF16;
  fa::FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  if (cu_seqlens) {
    if ((st = make_map_packed(&a.tmQ, Q, d, H, total, bf16)) != FA_OK) return st;
    if ((st = make_map_packed(&a.tmK, K, d, Hkv, total, bf16)) != FA_OK) return st;
    if ((st = make_map_packed(&a.tmV, V, d, Hkv, total, bf16)) != FA_OK) return st;
  } else {
    if ((st = make_map(&a.tmQ, Q, d, N, BH, bf16)) != FA_OK) return st;
    if ((st = make_map(&a.tmK, K, d, N, BHkv, bf16)) != FA_OK) return st;
    if ((st = make_map(&a.tmV, V, d, N, BHkv, bf16)) != FA_OK) return st;
  }
  if ((st = ctl_for_launch(&a.ctl)) != FA_OK) return st;
  a.cu_seqlens = cu_seqlens;
  a.H = H;
  a.total = total;
  a.O = O;
  a.L = L;
  a.N = N;
  a.BH = static_cast<int>(BH);
  a.group = H / Hkv;
  a.window = window < N ? window : 0;           // a window of N or more keys is plain causal
  a.c_log2 = scale * 1.4426950408889634f;
  cudaError_t e = fa::launch_fwd(a, d, bf16, causal != 0, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H,
                 int N, int d, int causal, float scale, fa_dtype dtype, void* stream) {
  return fwd_impl(Q, K, V, O, L, B, H, H, N, d, causal, scale, dtype, stream);
}

fa_status fa_fwd_gqa(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H,
                     int Hkv, int N, int d, int causal, float scale, fa_dtype dtype,
                     void* stream) {
  return fwd_impl(Q, K, V, O, L, B, H, Hkv, N, d, causal, scale, dtype, stream);
}

fa_status fa_fwd_swa(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H,
                     int Hkv, int N, int d, int window, float scale, fa_dtype dtype,
                     void* stream) {
  if (window < 1) return FA_ERR_INVALID_VALUE;
  return fwd_impl(Q, K, V, O, L, B, H, Hkv, N, d, 1, scale, dtype, stream, window);
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d, int causal) {
  if (check_common(B, H, N, d, causal, 1.0f, FA_FP16) != FA_OK) return 0;
  return fa::bwd_workspace_bytes(static_cast<long long>(B) * H, N, d);
}

static fa_status bwd_impl(const void* Q, const void* K, const void* V, const void* O,
                          const void* dO, const float* L, void* dQ, void* dK, void* dV,
                          void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int N,
                          int d, int causal, float scale, fa_dtype dtype, void* stream,
                          int window = 0, const int* cu_seqlens = nullptr, int total = 0) {
  fa_status st = check_common(B, H, N, d, causal, scale, static_cast<int>(dtype));
  if (st != FA_OK) return st;
  if ((st = check_heads(H, Hkv)) != FA_OK) return st;
  if (cu_seqlens && (st = check_packed(cu_seqlens, total)) != FA_OK) return st;
  if (!Q || !K || !V || !O || !dO || !L || !dQ || !dK || !dV) return FA_ERR_INVALID_VALUE;
  for (const void* p : {Q, K, V, O, dO, static_cast<const void*>(dQ), static_cast<const void*>(dK),
                        static_cast<const void*>(dV)})
    if (!aligned(p, 16)) return FA_ERR_MISALIGNED;
  if (!aligned(L, 4) || (workspace && !aligned(workspace, 16))) return FA_ERR_MISALIGNED;
  const long long BH = static_cast<long long>(B) * H;
  const size_t need = fa::bwd_workspace_bytes(BH, N, d);
  if (workspace && workspace_bytes < need) return FA_ERR_INVALID_VALUE;
  const long long BHkv = static_cast<long long>(B) * Hkv;
  const size_t rows = cu_seqlens ? static_cast<size_t>(total) : static_cast<size_t>(B) * N;
  const size_t nbytes = rows * H * d * 2, lbytes = rows * H * 4;
  const size_t kvbytes = rows * Hkv * d * 2;
  const void* outs[3] = {dQ, dK, dV};
  const size_t outsz[3] = {nbytes, kvbytes, kvbytes};
  const void* ins[5] = {Q, K, V, O, dO};
  const size_t insz[5] = {nbytes, kvbytes, kvbytes, nbytes, nbytes};
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 5; ++j)
      if (overlap(ins[j], insz[j], outs[i], outsz[i])) return FA_ERR_INVALID_VALUE;
    if (overlap(L, lbytes, outs[i], outsz[i])) return FA_ERR_INVALID_VALUE;
    for (int j = i + 1; j < 3; ++j)
      if (overlap(outs[i], outsz[i], outs[j], outsz[j])) return FA_ERR_INVALID_VALUE;
    if (workspace && overlap(workspace, need, outs[i], outsz[i])) return FA_ERR_INVALID_VALUE;
  }

  const bool bf16 = dtype == FA_BF16;
  fa::BwdArgs a;
  std::memset(&a, 0, sizeof(a));
  if (cu_seqlens) {
    if ((st = make_map_packed(&a.tmQ, Q, d, H, total, bf16)) != FA_OK) return st;
    if ((st = make_map_packed(&a.tmK, K, d, Hkv, total, bf16)) != FA_OK) return st;
    if ((st = make_map_packed(&a.tmV, V, d, Hkv, total, bf16)) != FA_OK) return st;
    if ((st = make_map_packed(&a.tmO, O, d, H, total, bf16)) != FA_OK) return st;
    if ((st = make_map_packed(&a.tmdO, dO, d, H, total, bf16)) != FA_OK) return st;
  } else {
    if ((st = make_map(&a.tmQ, Q, d, N, BH, bf16)) != FA_OK) return st;
    if ((st = make_map(&a.tmK, K, d, N, BHkv, bf16)) != FA_OK) return st;
    if ((st = make_map(&a.tmV, V, d, N, BHkv, bf16)) != FA_OK) return st;
    if ((st = make_map(&a.tmO, O, d, N, BH, bf16)) != FA_OK) return st;
    if ((st = make_map(&a.tmdO, dO, d, N, BH, bf16)) != FA_OK) return st;
  }
  if ((st = ctl_for_launch(&a.ctl)) != FA_OK) return st;
  a.cu_seqlens = cu_seqlens;
  a.H = H;
  a.total = total;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = workspace;
  bool owned = false;
  if (!ws) {
    cudaError_t e = cudaMallocAsync(&ws, need, s);
    if (e != cudaSuccess) return cuda_fail(e);
    owned = true;
  }
  a.Q = Q;
  a.O = O;
  a.dO = dO;
  a.L = L;
  a.Dvec = static_cast<float*>(ws);
  a.dQ = dQ;
  a.dK = dK;
  a.dV = dV;
  a.N = N;
  a.BH = static_cast<int>(BH);
  a.group = H / Hkv;
  a.window = window < N ? window : 0;           // a window of N or more keys is plain causal
  a.scale = scale;
  a.c_log2 = scale * 1.4426950408889634f;
  cudaError_t e = fa::launch_bwd(a, d, bf16, causal != 0, s);
  if (owned) {
    cudaError_t e2 = cudaFreeAsync(ws, s);
    if (e == cudaSuccess) e = e2;
  }
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* L, void* dQ, void* dK, void* dV, void* workspace,
                 size_t workspace_bytes, int B, int H, int N, int d, int causal, float scale,
                 fa_dtype dtype, void* stream) {
  return bwd_impl(Q, K, V, O, dO, L, dQ, dK, dV, workspace, workspace_bytes, B, H, H, N, d, causal,
                  scale, dtype, stream);
}

fa_status fa_bwd_gqa(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* L, void* dQ, void* dK, void* dV, void* workspace,
                     size_t workspace_bytes, int B, int H, int Hkv, int N, int d, int causal,
                     float scale, fa_dtype dtype, void* stream) {
  return bwd_impl(Q, K, V, O, dO, L, dQ, dK, dV, workspace, workspace_bytes, B, H, Hkv, N, d,
                  causal, scale, dtype, stream);
}

fa_status fa_bwd_swa(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* L, void* dQ, void* dK, void* dV, void* workspace,
                     size_t workspace_bytes, int B, int H, int Hkv, int N, int d, int window,
                     float scale, fa_dtype dtype, void* stream) {
  if (window < 1) return FA_ERR_INVALID_VALUE;
  return bwd_impl(Q, K, V, O, dO, L, dQ, dK, dV, workspace, workspace_bytes, B, H, Hkv, N, d, 1,
                  scale, dtype, stream, window);
}

fa_status fa_fwd_varlen(const void* Q, const void* K, const void* V, void* O, float* L,
                        const int* cu_seqlens, int B, int total, int max_seqlen, int H, int Hkv,
                        int d, int causal, int window, float scale, fa_dtype dtype, void* stream) {
  if (!cu_seqlens || window < 0 || (window > 0 && !causal)) return FA_ERR_INVALID_VALUE;
  return fwd_impl(Q, K, V, O, L, B, H, Hkv, max_seqlen, d, causal, scale, dtype, stream, window,
                  cu_seqlens, total);
}

size_t fa_bwd_varlen_workspace_size(int B, int max_seqlen, int H, int d) {
  return fa_bwd_workspace_size(B, H, max_seqlen, d, 1);
}

fa_status fa_bwd_varlen(const void* Q, const void* K, const void* V, const void* O,
                        const void* dO, const float* L, void* dQ, void* dK, void* dV,
                        void* workspace, size_t workspace_bytes, const int* cu_seqlens, int B,
                        int total, int max_seqlen, int H, int Hkv, int d, int causal, int window,
                        float scale, fa_dtype dtype, void* stream) {
  if (!cu_seqlens || window < 0 || (window > 0 && !causal)) return FA_ERR_INVALID_VALUE;
  return bwd_impl(Q, K, V, O, dO, L, dQ, dK, dV, workspace, workspace_bytes, B, H, Hkv, max_seqlen,
                  d, causal, scale, dtype, stream, window, cu_seqlens, total);
}

// Forward on 8-bit E4M3 inputs with per-tensor descale factors (d = 128).
fa_status fa_fwd_fp8(const void* Q8, const void* K8, const void* Vt8, void* O, float* L, int B,
                     int H, int Hkv, int N, int d, int causal, float scale, float q_scale,
                     float k_scale, float v_scale, void* stream) {
  fa_status st = check_common(B, H, N, d, causal, scale, FA_BF16);
  if (st != FA_OK) return st;
  if ((st = check_heads(H, Hkv)) != FA_OK) return st;
  for (float x : {q_scale, k_scale, v_scale})
    if (!(std::isfinite(x) && x > 0.f)) return FA_ERR_INVALID_VALUE;
  if (d != 128 || N % 16 != 0) return FA_ERR_UNSUPPORTED;
  if (!Q8 || !K8 || !Vt8 || !O || !L) return FA_ERR_INVALID_VALUE;
  if (!aligned(Q8, 16) || !aligned(K8, 16) || !aligned(Vt8, 16) || !aligned(O, 16) ||
      !aligned(L, 4))
    return FA_ERR_MISALIGNED;
  const long long BH = static_cast<long long>(B) * H, BHkv = static_cast<long long>(B) * Hkv;
  const size_t qbytes = static_cast<size_t>(BH) * N * d, kvbytes = static_cast<size_t>(BHkv) * N * d;
  const size_t obytes = qbytes * 2, lbytes = static_cast<size_t>(BH) * N * 4;
  const void* ins[3] = {Q8, K8, Vt8};
  const size_t insz[3] = {qbytes, kvbytes, kvbytes};
  for (int i = 0; i < 3; ++i)
    if (overlap(ins[i], insz[i], O, obytes) || overlap(ins[i], insz[i], L, lbytes))
      return FA_ERR_INVALID_VALUE;
  if (overlap(O, obytes, L, lbytes)) return FA_ERR_INVALID_VALUE;
  fa::Fwd8Args a;
  std::memset(&a, 0, sizeof(a));
  if ((st = make_map_bytes(&a.tmQ, Q8, d, N, BH)) != FA_OK) return st;
  if ((st = make_map_bytes(&a.tmK, K8, d, N, BHkv)) != FA_OK) return st;
  if ((st = make_map_bytes(&a.tmVt, Vt8, N, d, BHkv)) != FA_OK) return st;
  if ((st = ctl_for_launch(&a.ctl)) != FA_OK) return st;
  a.O = O;
  a.L = L;
  a.N = N;
  a.BH = static_cast<int>(BH);
  a.group = H / Hkv;
  a.c_log2 = scale * q_scale * k_scale * 1.4426950408889634f;
  a.o_scale = v_scale;
  cudaError_t e = fa::launch_fwd8(a, causal != 0, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

fa_status fa_quantize_fp8(const void* X, void* X8, long long mats, int rows, int cols,
                          float inv_scale, int transpose, fa_dtype dtype, void* stream) {
  if (mats < 1 || rows < 1 || cols < 1 || (transpose != 0 && transpose != 1))
    return FA_ERR_INVALID_VALUE;
  if (!(std::isfinite(inv_scale) && inv_scale > 0.f)) return FA_ERR_INVALID_VALUE;
  if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if (transpose && (mats > 65535 || (rows + 31) / 32 > 65535)) return FA_ERR_UNSUPPORTED;
  if (!X || !X8) return FA_ERR_INVALID_VALUE;
  if (!aligned(X, 2)) return FA_ERR_MISALIGNED;
  const size_t n = static_cast<size_t>(mats) * rows * cols;
  if (overlap(X, n * 2, X8, n)) return FA_ERR_INVALID_VALUE;
  cudaError_t e = fa::launch_quant8(X, X8, mats, rows, cols, inv_scale, transpose != 0,
                                    dtype == FA_BF16, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

// Split-KV decoding: one query row per (batch, head) against the first
// cache_seqlens[b] rows of K/V caches (B, Hkv, Nmax, d).
size_t fa_decode_workspace_size(int B, int H, int Hkv, int Nmax, int d) {
  if (check_common(B, H, Nmax, d, 0, 1.0f, FA_FP16) != FA_OK || check_heads(H, Hkv) != FA_OK)
    return 0;
  int chunk = 0;
  const int splits = fa::decode_parts(B, H, Hkv, Nmax, &chunk);
  return static_cast<size_t>(B) * H * splits * (d + 4) * sizeof(float);
}

static fa_status decode_impl(const void* Q, const void* Kc, const void* Vc,
                             const int* cache_seqlens, void* O, float* L, void* workspace,
                             size_t workspace_bytes, int B, int H, int Hkv, int Nmax, int d,
                             float scale, fa_dtype dtype, void* stream, bool c8, float k_scale,
                             float v_scale) {
  fa_status st = check_common(B, H, Nmax, d, 0, scale, static_cast<int>(dtype));
  if (st != FA_OK) return st;
  if ((st = check_heads(H, Hkv)) != FA_OK) return st;
  if (Nmax > (1 << 30)) return FA_ERR_UNSUPPORTED;
  if (!Q || !Kc || !Vc || !cache_seqlens || !O || !L) return FA_ERR_INVALID_VALUE;
  if (!aligned(Q, 16) || !aligned(Kc, 16) || !aligned(Vc, 16) || !aligned(O, 16) ||
      !aligned(L, 4) || !aligned(cache_seqlens, 4) || (workspace && !aligned(workspace, 16)))
    return FA_ERR_MISALIGNED;
  int chunk = 0;
  const int splits = fa::decode_parts(B, H, Hkv, Nmax, &chunk);
  const long long ctas = static_cast<long long>(B) * Hkv * splits *
                         ((H / Hkv) / fa::decode_rows(H, Hkv));
  if (ctas > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  const size_t need = fa_decode_workspace_size(B, H, Hkv, Nmax, d);
  if (workspace && workspace_bytes < need) return FA_ERR_INVALID_VALUE;
  const size_t qbytes = static_cast<size_t>(B) * H * d * 2, lbytes = static_cast<size_t>(B) * H * 4;
  const size_t cbytes = static_cast<size_t>(B) * Hkv * Nmax * d * (c8 ? 1 : 2);
  const void* ins[4] = {Q, Kc, Vc, cache_seqlens};
  const size_t insz[4] = {qbytes, cbytes, cbytes, static_cast<size_t>(B) * 4};
  for (int i = 0; i < 4; ++i) {
    if (overlap(ins[i], insz[i], O, qbytes) || overlap(ins[i], insz[i], L, lbytes))
      return FA_ERR_INVALID_VALUE;
    if (workspace && overlap(ins[i], insz[i], workspace, need)) return FA_ERR_INVALID_VALUE;
  }
  if (overlap(O, qbytes, L, lbytes)) return FA_ERR_INVALID_VALUE;
  if (workspace && (overlap(workspace, need, O, qbytes) || overlap(workspace, need, L, lbytes)))
    return FA_ERR_INVALID_VALUE;

  const bool bf16 = dtype == FA_BF16;
  fa::DecodeArgs a;
  std::memset(&a, 0, sizeof(a));
  const long long BHkv = static_cast<long long>(B) * Hkv;
  const int rows = fa::decode_key_rows(d, c8);
  if (c8) {
    if ((st = make_map_bytes(&a.tmK, Kc, d, Nmax, BHkv, rows)) != FA_OK) return st;
    if ((st = make_map_bytes(&a.tmV, Vc, d, Nmax, BHkv, rows)) != FA_OK) return st;
  } else {
    if ((st = make_map(&a.tmK, Kc, d, Nmax, BHkv, bf16, rows)) != FA_OK) return st;
    if ((st = make_map(&a.tmV, Vc, d, Nmax, BHkv, bf16, rows)) != FA_OK) return st;
  }
  if ((st = ctl_for_launch(&a.ctl)) != FA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = workspace;
  bool owned = false;
  if (!ws) {
    cudaError_t e = cudaMallocAsync(&ws, need, s);
    if (e != cudaSuccess) return cuda_fail(e);
    owned = true;
  }
  a.Q = Q;
  a.seqlens = cache_seqlens;
  a.O = O;
  a.L = L;
  a.part = static_cast<float*>(ws);
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.Nmax = Nmax;
  a.n_splits = splits;
  a.chunk = chunk;
  a.c_log2 = scale * (c8 ? k_scale : 1.f) * 1.4426950408889634f;
  a.o_scale = c8 ? v_scale : 1.f;
  cudaError_t e = fa::launch_decode(a, d, bf16, c8, s);
  if (owned) {
    cudaError_t e2 = cudaFreeAsync(ws, s);
    if (e == cudaSuccess) e = e2;
  }
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

fa_status fa_decode(const void* Q, const void* Kc, const void* Vc, const int* cache_seqlens,
                    void* O, float* L, void* workspace, size_t workspace_bytes, int B, int H,
                    int Hkv, int Nmax, int d, float scale, fa_dtype dtype, void* stream) {
  return decode_impl(Q, Kc, Vc, cache_seqlens, O, L, workspace, workspace_bytes, B, H, Hkv, Nmax,
                     d, scale, dtype, stream, false, 1.f, 1.f);
}

fa_status fa_decode_fp8(const void* Q, const void* Kc8, const void* Vc8, const int* cache_seqlens,
                        void* O, float* L, void* workspace, size_t workspace_bytes, int B, int H,
                        int Hkv, int Nmax, int d, float scale, float k_scale, float v_scale,
                        fa_dtype dtype, void* stream) {
  for (float x : {k_scale, v_scale})
    if (!(std::isfinite(x) && x > 0.f)) return FA_ERR_INVALID_VALUE;
  if (d != 128 && check_common(B, H, Nmax, d, 0, scale, static_cast<int>(dtype)) == FA_OK)
    return FA_ERR_UNSUPPORTED;
  return decode_impl(Q, Kc8, Vc8, cache_seqlens, O, L, workspace, workspace_bytes, B, H, Hkv,
                     Nmax, d, scale, dtype, stream, true, k_scale, v_scale);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Backward without allocation.  Some callers cannot call cudaMalloc at all:
// plugins of a host framework that owns every byte of device memory, and
// deployments that hand the library a fixed memory budget up front.  They get
// fa_bwd_noalloc, whose scratch lives in this file-scope array instead of a
// workspace: every GPU that loads the library holds it until the process exits.
static constexpr size_t kNoAllocScratchBytes = 16u << 20;   // 16 MiB
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

// Device address of the scratch array in the current context.  On the host the
// array's name is only a stand-in, never a device address, so it is looked up in the
// current context (once per context) and the looked-up pointer is what the kernels
// receive.
static fa_status noalloc_scratch(float** out) {
  void* p = nullptr;
  fa_status st = symbol_address(reinterpret_cast<const void*>(&g_noalloc_scratch), &p);
  if (st != FA_OK) return st;
  *out = static_cast<float*>(p);
  return FA_OK;
}

extern "C" {

fa_status fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                         const void* dO, const float* L, void* dQ, void* dK, void* dV, int B,
                         int H, int N, int d, int causal, float scale, fa_dtype dtype,
                         void* stream) {
  fa_status st = check_common(B, H, N, d, causal, scale, static_cast<int>(dtype));
  if (st != FA_OK) return st;
  const size_t need = fa::bwd_workspace_bytes(static_cast<long long>(B) * H, N, d);
  if (need > kNoAllocScratchBytes) return FA_ERR_UNSUPPORTED;   // more than the static scratch
  float* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != FA_OK) return st;
  // Same validation and kernels as fa_bwd, with the static array as its workspace;
  // a non-NULL workspace means fa_bwd allocates nothing.
  return fa_bwd(Q, K, V, O, dO, L, dQ, dK, dV, scratch, kNoAllocScratchBytes, B, H, N, d, causal,
                scale, dtype, stream);
}

}  // extern "C"
