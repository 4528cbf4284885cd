/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library.
 *
 * The operation is exact scaled-dot-product attention computed tile by tile
 * with an online softmax, forward and backward ("flash-attn-triton" docs page:
 * sections "The argument", "Tiling softmax is exact algebra" with Fig. 3, and
 * "Scope"; FlashAttention note, "Key Mechanisms").  For each (batch b, head h):
 *
 *     S = scale * Q K^T                     (N x N, never stored)
 *     causal: key j is allowed for query i iff j <= i (lower triangle)
 *     P = softmax over the allowed keys of each row
 *     O = P V
 *     L = logsumexp of the allowed scaled scores of each row (natural log)
 *
 * and the backward returns dQ, dK, dV for an upstream gradient dO, rebuilding P
 * from the saved L instead of storing it (docs page, "Scope"; FlashAttention
 * note, "Key Mechanisms", backward recomputation).
 *
 * Conventions shared by every call
 *   Layout     Q, K, V, O, dO, dQ, dK, dV: dense row-major (B, H, N, d) arrays of
 *              16-bit floats (fp16 or bf16, all the same); element (b,h,n,c) at
 *              ((b*H + h)*N + n)*d + c.  L: dense (B, H, N) fp32.
 *   Memory     every pointer is CUDA device memory (or managed memory) of the
 *              current device; the caller owns every buffer; the library keeps
 *              no pointer after a call returns.  Outputs must not overlap inputs.
 *   Alignment  16-bit arrays and the workspace: 16-byte aligned; L: 4-byte aligned.
 *   Streams    `stream` is a cudaStream_t (NULL = the legacy default stream).
 *              Calls only enqueue work: they return before the GPU finishes and
 *              never synchronise, except fa_device_status.  So a sequence of calls
 *              can be captured into a CUDA graph once each call has run eagerly
 *              (the first call of a kind sets kernel attributes) and, for the
 *              backward, with a caller workspace; the replay gives the eager
 *              results bit for bit.
 *   Errors     arguments are validated before anything is launched; a call that
 *              returns an error has enqueued nothing (launch failures excepted:
 *              FA_ERR_CUDA, with the CUDA error code from fa_last_cuda_error()).
 *   Supported  d in {32, 64, 128}; fp16 or bf16; causal 0/1; any N >= 1 (N need
 *              not be a multiple of the 128-row tile); scale finite and > 0.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_VALUE = 1,  /* NULL pointer, B/H/N < 1, bad scale, short workspace, overlap */
  FA_ERR_UNSUPPORTED = 2,    /* d not in {32,64,128}, unknown dtype, sizes beyond the limits */
  FA_ERR_MISALIGNED = 3,     /* a pointer violates the alignment rule above */
  FA_ERR_CUDA = 4,           /* a CUDA runtime/driver call or a launch failed */
  FA_ERR_TIMEOUT = 5         /* a kernel gave up a bounded wait (see fa_device_status) */
} fa_status;

typedef enum fa_dtype { FA_FP16 = 0, FA_BF16 = 1 } fa_dtype;

/* Forward.  Writes O (B,H,N,d) and L (B,H,N) fp32 = natural-log logsumexp of the
 * allowed scaled scores of each row (docs page Fig. 3: L = m + log l, one float
 * per row, the only state the backward needs).  Q, K, V are read once per
 * 128-query-row tile pair; the N x N score matrix never reaches memory. */
fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* L,
                 int B, int H, int N, int d, int causal, float scale, fa_dtype dtype,
                 void* stream);

/* Bytes of device workspace fa_bwd needs for these sizes: the per-row delta
 * D = rowsum(dO o O) and L * log2(e), both fp32, padded to whole 128-row tiles.
 * Returns 0 for sizes fa_bwd would reject. */
size_t fa_bwd_workspace_size(int B, int H, int N, int d, int causal);

/* Backward.  Given Q, K, V, the forward's O and L, and dO, writes dQ, dK, dV
 * (16-bit, same layout as Q).  P is rebuilt from L (docs page, "Scope"):
 *   dV = P^T dO, dP = dO V^T, D = rowsum(dO o O), dS = P o (dP - D),
 *   dQ = scale dS K, dK = scale dS^T Q.
 * `workspace` is device memory of at least fa_bwd_workspace_size() bytes, used
 * as scratch during the call; pass NULL to let the library take it from the
 * stream-ordered allocator (cudaMallocAsync / cudaFreeAsync on `stream`). */
fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* L, void* dQ, void* dK, void* dV, void* workspace,
                 size_t workspace_bytes, int B, int H, int N, int d, int causal, float scale,
                 fa_dtype dtype, void* stream);

/* Grouped-query and multi-query attention (GQA / MQA).  The docs page lists
 * "MQA/GQA" among the features its kernels do not have yet ("Scope"); the note
 * credits FlashAttention-2 with adding them ("Versions and Evolution").  K and V
 * have Hkv heads instead of H: query head h of batch b attends with K/V head
 * h / (H/Hkv) of batch b (consecutive query heads share one K/V head; Hkv == 1 is
 * MQA, Hkv == H is fa_fwd / fa_bwd).  Each query head computes exactly what
 * fa_fwd computes with that K/V head; in the backward, dK and dV of a shared head
 * are the sums over its H/Hkv query heads.
 *   Layout   Q, O, dO, dQ: (B, H, N, d); K, V, dK, dV: (B, Hkv, N, d); L: (B, H, N).
 *   Errors   as fa_fwd / fa_bwd, plus FA_ERR_INVALID_VALUE when Hkv < 1, Hkv > H
 *            or H is not a multiple of Hkv.
 *   Workspace of fa_bwd_gqa: fa_bwd_workspace_size(B, H, N, d, causal) bytes (it
 *            depends on the query heads only), or NULL as for fa_bwd. */
fa_status fa_fwd_gqa(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H,
                     int Hkv, int N, int d, int causal, float scale, fa_dtype dtype,
                     void* stream);
fa_status fa_bwd_gqa(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* L, void* dQ, void* dK, void* dV, void* workspace,
                     size_t workspace_bytes, int B, int H, int Hkv, int N, int d, int causal,
                     float scale, fa_dtype dtype, void* stream);

/* Sliding-window (local) attention: causal, each query sees only the `window`
 * most recent keys, itself included: key j is allowed for query i iff
 * i - window < j <= i.  The docs page lists sliding windows among the features its
 * kernels do not have yet ("Scope") and fixes no convention; this causal band is
 * the plain reading.  Hkv as for fa_fwd_gqa (Hkv == H: no sharing).  window >=
 * N is plain causal attention.  Only the KV tiles inside the band are computed.
 *   Errors   as fa_fwd_gqa / fa_bwd_gqa, plus FA_ERR_INVALID_VALUE for window < 1.
 *   Workspace of fa_bwd_swa: fa_bwd_workspace_size(B, H, N, d, 1), or NULL. */
fa_status fa_fwd_swa(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H,
                     int Hkv, int N, int d, int window, float scale, fa_dtype dtype,
                     void* stream);
fa_status fa_bwd_swa(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* L, void* dQ, void* dK, void* dV, void* workspace,
                     size_t workspace_bytes, int B, int H, int Hkv, int N, int d, int window,
                     float scale, fa_dtype dtype, void* stream);

/* Variable-length batches: B sequences of different lengths packed one after
 * another (the docs page lists "variable-length batches" among the features its
 * kernels do not have yet, "Scope").  Sequence b holds rows cu_seqlens[b] ..
 * cu_seqlens[b+1]-1 of every tensor and attends only to its own keys (causal and
 * window as in fa_fwd / fa_fwd_swa, measured from the sequence's first row; window
 * 0 = none; window > 0 needs causal); K/V heads shared as in fa_fwd_gqa.
 *   Layout   Q, O, dO, dQ: (total, H, d); K, V, dK, dV: (total, Hkv, d), rows
 *            row-major with heads inside a row; L: (H, total) fp32.
 *   cu_seqlens  device int32 [B+1]: 0 = cu[0] <= cu[1] <= ... <= cu[B] = total.
 *            max_seqlen >= every cu[b+1] - cu[b] (it sizes the grid).  The kernels
 *            clamp every sequence to rows [0, total) and to max_seqlen rows, so
 *            offsets that break these rules leave rows uncomputed but never make a
 *            kernel touch memory outside the tensors.
 *   Workspace of fa_bwd_varlen: fa_bwd_varlen_workspace_size(B, max_seqlen, H, d),
 *            or NULL.
 *   Errors   as fa_fwd_gqa / fa_bwd_gqa (max_seqlen in the role of N), plus
 *            FA_ERR_INVALID_VALUE for cu_seqlens NULL, total < 1, window < 0 or a
 *            window without causal; FA_ERR_MISALIGNED if cu_seqlens is not 4-byte
 *            aligned. */
fa_status fa_fwd_varlen(const void* Q, const void* K, const void* V, void* O, float* L,
                        const int* cu_seqlens, int B, int total, int max_seqlen, int H, int Hkv,
                        int d, int causal, int window, float scale, fa_dtype dtype, void* stream);
size_t fa_bwd_varlen_workspace_size(int B, int max_seqlen, int H, int d);
fa_status fa_bwd_varlen(const void* Q, const void* K, const void* V, const void* O,
                        const void* dO, const float* L, void* dQ, void* dK, void* dV,
                        void* workspace, size_t workspace_bytes, const int* cu_seqlens, int B,
                        int total, int max_seqlen, int H, int Hkv, int d, int causal, int window,
                        float scale, fa_dtype dtype, void* stream);

/* Forward on 8-bit E4M3 inputs (the FP8 precision that the FlashAttention note
 * credits to FlashAttention-3, "Versions and Evolution"), head dim 128.  The
 * inputs are E4M3 codes with per-tensor descale factors: the result is the
 * attention of q_scale*Q, k_scale*K and v_scale*V, computed as the 16-bit
 * forward does ("flash-attn-triton" docs page, Fig. 3) with both products on the
 * tensor cores in 8 bits: S = Q K^T from the codes (fp32 accumulation), and
 * O += P V with P rounded to E4M3 (p <= 2^8 by the running-max rule); the sum l
 * is taken over the unrounded p.
 *   Q8     (B, H, N, 128) codes, one byte each.
 *   K8     (B, Hkv, N, 128) codes.
 *   Vt8    (B, Hkv, 128, N) codes of V with its last two axes swapped (see
 *          fa_quantize_fp8).
 *   O      (B, H, N, 128) bf16 output.  L (B, H, N) fp32, natural log, of the
 *          scores scale * q_scale * k_scale * (Q8 . K8).
 *   Query head h uses K/V head h / (H / Hkv).  N must be a multiple of 16 (the
 *   rows of Vt8 are N bytes apart and TMA wants 16-byte strides).  Q8, K8, Vt8
 *   and O 16-byte aligned, L 4-byte aligned.
 *   Errors: FA_ERR_UNSUPPORTED for d != 128 or N % 16 != 0; FA_ERR_INVALID_VALUE
 *   for NULL pointers, bad sizes, H not a multiple of Hkv, non-positive or
 *   non-finite scale or descale factors, overlapping buffers; FA_ERR_MISALIGNED
 *   for the alignment rules.  Asynchronous on `stream`. */
fa_status fa_fwd_fp8(const void* Q8, const void* K8, const void* Vt8, void* O, float* L, int B,
                     int H, int Hkv, int N, int d, int causal, float scale, float q_scale,
                     float k_scale, float v_scale, void* stream);

/* E4M3 codes of X * inv_scale, rounded to nearest even and saturated at +-448
 * (the preparation step of fa_fwd_fp8: inv_scale is 1 / descale).  X holds `mats`
 * row-major rows x cols matrices of 16-bit values (dtype FA_FP16 / FA_BF16); X8
 * receives one byte per element, each matrix transposed (cols x rows) when
 * transpose = 1.  Errors: FA_ERR_INVALID_VALUE for NULL pointers, sizes < 1, a
 * non-positive or non-finite inv_scale or overlapping buffers;
 * FA_ERR_UNSUPPORTED for another dtype, or with transpose for more than 65535
 * matrices or 2^21 rows; FA_ERR_MISALIGNED if X is not 2-byte aligned.
 * Asynchronous on `stream`. */
fa_status fa_quantize_fp8(const void* X, void* X8, long long mats, int rows, int cols,
                          float inv_scale, int transpose, fa_dtype dtype, void* stream);

/* Split-KV decoding: one new query row per (batch, head) attends to the first
 * cache_seqlens[b] cached keys of its sequence.  The key range is cut into
 * pieces whose softmax partial states (running max m, sum l, unnormalised
 * output acc) are merged exactly on the GPU: the tutorial page "What is
 * FlashAttention?", "Softmax in pieces" (merging two partial results), applied
 * to a key/value cache (the FlashAttention note lists inference serving with a
 * KV cache among the method's uses: "Applications and Use Cases").
 *   Q            (B, H, d) fp16/bf16, one query row per head.
 *   Kc, Vc       (B, Hkv, Nmax, d) caches; rows at and past cache_seqlens[b]
 *                are never used (their contents may be anything).
 *   cache_seqlens  device int32 [B]; values are clamped to [0, Nmax].  A
 *                sequence with no cached key gets O = 0, L = -inf.
 *   O            (B, H, d) output, same dtype.
 *   L            (B, H) fp32, the natural-log logsumexp of each row's scores.
 *   workspace    fa_decode_workspace_size(B, H, Hkv, Nmax, d) bytes of device
 *                memory (16-byte aligned) for the partial states, or NULL: the
 *                library then allocates and frees it on `stream`.
 *   Query head h uses K/V head h / (H / Hkv).  Q, Kc, Vc and O 16-byte aligned.
 *   Errors: FA_ERR_INVALID_VALUE for NULL pointers, B, H or Nmax < 1, H not a
 *   multiple of Hkv, a non-positive or non-finite scale, a short workspace or
 *   overlapping buffers; FA_ERR_UNSUPPORTED for d not 32/64/128, another dtype,
 *   Nmax above 2^30 or sizes past the index limits; FA_ERR_MISALIGNED for the
 *   alignment rules.
 *   Asynchronous on `stream`; nothing is read back. */
size_t fa_decode_workspace_size(int B, int H, int Hkv, int Nmax, int d);
fa_status fa_decode(const void* Q, const void* Kc, const void* Vc, const int* cache_seqlens,
                    void* O, float* L, void* workspace, size_t workspace_bytes, int B, int H,
                    int Hkv, int Nmax, int d, float scale, fa_dtype dtype, void* stream);

/* Split-KV decoding from 8-bit E4M3 caches with per-tensor descale factors: as
 * fa_decode, with Kc8 and Vc8 (B, Hkv, Nmax, d) holding one E4M3 code per value,
 * standing for k_scale * K and v_scale * V (the FP8 precision of the FlashAttention
 * note's FlashAttention-3 entry, "Versions and Evolution", applied to a decoding
 * cache).  The scores are formed in fp32 from the decoded codes and P stays fp32,
 * so only the cache is in 8 bits.  Q, O in fp16/bf16 (dtype), L fp32 as in
 * fa_decode; the workspace is fa_decode_workspace_size(B, H, Hkv, Nmax, d) bytes or
 * NULL.  d must be 128 (FA_ERR_UNSUPPORTED otherwise); k_scale and v_scale must be
 * positive and finite (FA_ERR_INVALID_VALUE); the other errors are fa_decode's. */
fa_status fa_decode_fp8(const void* Q, const void* Kc8, const void* Vc8, const int* cache_seqlens,
                        void* O, float* L, void* workspace, size_t workspace_bytes, int B, int H,
                        int Hkv, int Nmax, int d, float scale, float k_scale, float v_scale,
                        fa_dtype dtype, void* stream);

/* Static description of a status code. */
const char* fa_status_string(fa_status s);

/* CUDA error code (a cudaError_t value) behind the last FA_ERR_CUDA returned on
 * the calling thread; 0 if none. */
int fa_last_cuda_error(void);

/* Synchronises `stream`, then reads and clears the current device's status
 * word: FA_ERR_TIMEOUT if any kernel of this library gave up a bounded wait
 * since the last read; FA_ERR_UNSUPPORTED if a kernel found its dynamic shared
 * memory not aligned to 1024 bytes and skipped its work (not expected on
 * sm_103a); FA_OK otherwise (FA_ERR_CUDA if the read failed). */
fa_status fa_device_status(void* stream);

/* Bound, in nanoseconds, on any single wait inside the kernels (default 2 s).
 * ns == 0 restores the default.  Applies to launches made after the call. */
fa_status fa_set_wait_limit_ns(unsigned long long ns);

/* Failure-detection self test: launches one CTA that waits on a barrier nothing
 * will complete, bounded by `limit_ns`; the kernel records a timeout and exits.
 * Synchronises `stream` and returns what fa_device_status then reports
 * (FA_ERR_TIMEOUT when the bound works).  Faults nothing. */
fa_status fa_selftest_timeout(unsigned long long limit_ns, void* stream);

/* Per-kernel timing trace (the method's own benchmark harness measures speed
 * and TFLOP/s: docs page, "Scope" and Table 3).  While enabled, every kernel
 * launch of this library is bracketed by two CUDA events recorded on its
 * stream, from a fixed pool of 4096 launches (later launches are not traced).
 * fa_trace_enable(1) (re)starts recording and clears earlier records (the
 * first call creates the events); fa_trace_enable(0) stops it.  Not
 * thread-safe: trace from one host thread. */
fa_status fa_trace_enable(int on);

/* Name of trace kind `kind` (0: forward kernel, 1: backward pre-pass, 2:
 * backward dK/dV kernel, 3: backward dQ kernel, 4: decode split kernel, 5:
 * decode merge kernel, 6: FP8 forward kernel); NULL when out of range. */
const char* fa_trace_kind_name(int kind);

/* Waits for the recorded events of kind `kind`, then writes the summed GPU
 * time in milliseconds and the number of traced launches. */
fa_status fa_trace_read(int kind, double* total_ms, long long* launches);

/* Backward that allocates nothing.  The pages have no counterpart: this entry
 * exists for callers, not for the method.  Some callers cannot call cudaMalloc
 * at all -- a plugin inside a host framework that owns every byte of device
 * memory, or a deployment handed a fixed memory budget up front -- and fa_bwd
 * either takes a caller workspace or allocates one.  fa_bwd_noalloc computes
 * what fa_bwd computes, with the same arguments minus the workspace.  Its
 * scratch is a 16 MiB device array inside the library, held by every GPU that
 * loads the library until the process exits; sizes whose scratch need
 * (fa_bwd_workspace_size) exceeds 16 MiB are rejected with FA_ERR_UNSUPPORTED
 * before anything is launched.  The first call in a CUDA context looks up the
 * array's device address there (cudaGetSymbolAddress, with the caller's device and
 * context current; a context destroyed and recreated, e.g. by cudaDeviceReset, is
 * looked up again); make that first call before any stream capture.  The lookup is
 * guarded by a lock, so first calls from several host threads are safe.  All
 * calls share the one array and it keeps the last call's contents: calls that
 * overlap on the GPU (other streams, other host threads) race on it, so
 * serialise them.  Nothing in it
 * needs to start at zero: each call writes every scratch value before reading
 * it.  Capacity: 8 bytes per row, B*H*ceil(N/128)*128 up to 2,097,152 rows. */
fa_status fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                         const void* dO, const float* L, void* dQ, void* dK, void* dV, int B,
                         int H, int N, int d, int causal, float scale, fa_dtype dtype,
                         void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
