/*
 * fa.h — C ABI of the GB300 (sm_103a) exact-attention library.
 *
 * Operation (all entry points): exact scaled-dot-product attention,
 *     O = softmax(scale * Q K^T + M) V,    LSE_i = ln sum_j exp(scale * (Q K^T)_ij + M_ij)
 * where M is 0, or -inf above the bottom-right-aligned diagonal when causal
 * (key j is visible to query i iff j <= i + (Sk - Sq)). The result is the exact
 * one: the kernels tile the computation with an online softmax and never write
 * the score matrix to memory ("FlashAttention-4 Conquers Asymmetric GPU
 * Hardware Scaling", episode description, lineage paragraph; the method's
 * kernel design is the one summarised in "FlashAttention-4: Algorithm and Kernel
 * Pipelining Co-Design for Asymmetric Hardware Scaling", abstract and Summary).
 * Query heads share key/value heads in groups of Hq / Hkv (grouped-query
 * attention); query head h uses KV head h / (Hq / Hkv).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers to contiguous memory on the
 *     current CUDA device; base addresses must be 16-byte aligned.
 *   - bf16 = IEEE bfloat16 (2 bytes); fp32 = IEEE binary32.
 *   - Dense layout: q, o, dout, dq are [B][Sq][Hq][d]; k, v, dk, dv are
 *     [B][Sk][Hkv][d]; lse is fp32 [B][Hq][Sq].
 *   - Packed variable-length layout (cu_seqlens != NULL): B is the number of
 *     sequences, cu_seqlens is a DEVICE int32 array of B+1 non-decreasing
 *     offsets with cu_seqlens[0] = 0, and Sq == Sk == cu_seqlens[B] = T, the
 *     number of packed rows. q, o, dout, dq are [T][Hq][d]; k, v, dk, dv are
 *     [T][Hkv][d]; lse is fp32 [Hq][T]. Sequence i owns rows
 *     [cu_seqlens[i], cu_seqlens[i+1]) of every tensor (self-attention: one
 *     boundary list for queries and keys).
 *   - d (head dimension) is 64, 128, 192 or 256; scale must be finite and > 0.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream). FA_OK means "validated and enqueued". The library allocates no
 *     memory on any call and keeps no per-call state; the caller owns all
 *     buffers and must keep them alive until the stream work completes.
 *   - Rows with no visible key (possible only when causal with Sq > Sk) get
 *     O = 0 and LSE = +inf, which makes their backward contribution zero.
 *   - Errors are returned as fa_status codes; nothing is thrown across the ABI.
 *     fa_last_error() returns a thread-local message for the last failure.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* bad pointer, size, alignment or layout */
  FA_ERR_UNSUPPORTED = 2,  /* valid but not supported (e.g. a head dim not listed) */
  FA_ERR_ARCH = 3,         /* current device is not compute capability 10.3 */
  FA_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed; see fa_last_error() */
  FA_ERR_WORKSPACE = 5,    /* backward workspace missing or too small */
  FA_ERR_TIMEOUT = 6       /* a kernel's bounded wait expired (see fa_get_device_error) */
} fa_status;

/*
 * Forward: O (bf16) and LSE (fp32, natural log of the scaled scores).
 *   q [.., Hq, d], k/v [.., Hkv, d] bf16 inputs (read only); o bf16 output,
 *   lse fp32 output (layouts above). Hq % Hkv == 0. Sq, Sk >= 0 (0 = nothing
 *   to do). The kernel is one persistent launch ordering its work
 *   longest-first (LPT) for causal and packed batches.
 */
FA_API int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
           int Hkv, int Sq, int Sk, int d, int causal, float scale, const int* cu_seqlens,
           void* stream);

/*
 * FP8 (e4m3) quantization of a bf16 attention input x [B, S, H, d] (device,
 * 16-byte aligned; d = 64 or 128) for fa_fwd_fp8. The FlashAttention-4 pages
 * name low precision only through the FlashAttention-3 title (their reference
 * lists); the scaling below is this library's reading:
 *   layout 0 (Q, K): codes [B, S, H, d] (1 byte each); scales float
 *     [B, H, ceil(S/128)], one per 128-row block over its rows and d columns.
 *   layout 1 (V): codes transposed, [B, H, d, S_pad] with S_pad = S rounded
 *     up to 16 (the pad holds zero codes); scales float [B, H].
 * scale = amax / 448 (1 if amax = 0); code = e4m3(x * r) with r = 1 / scale
 * (scale, r and each product rounded to float32), round to nearest even,
 * saturating at +-448. Runs on `stream`
 * (layout 1: a memset and three kernels, with `scales` as their scratch).
 * Errors: FA_ERR_INVALID_ARG (NULL or misaligned pointer, bad sizes or
 * layout), FA_ERR_UNSUPPORTED (d), FA_ERR_CUDA.
 */
FA_API int fa_quantize_fp8(const void* x, int B, int S, int H, int d, int layout, void* codes,
                           float* scales, void* stream);

/*
 * FP8 forward: O (bf16 [B, Sq, Hq, d]) and LSE (fp32 [B, Hq, Sq]) of exact
 * attention over the dequantized inputs Q^ = code * q_scale etc., from the
 * outputs of fa_quantize_fp8 (q8, k8 layout 0 with [B, Sq, Hq, d] and
 * [B, Sk, Hkv, d]; vt8 layout 1, [B, Hkv, d, Sk_pad]). Same masking, GQA and
 * LSE conventions as fa_fwd (dense layouts, d = 128). Both products run on the
 * tensor cores in e4m3 with fp32 accumulation; the softmax weights are rounded
 * to e4m3 for the P V product, so O carries that rounding (relative error of
 * each weight <= 2^-4) while the LSE does not. Errors as fa_fwd.
 */
FA_API int fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_scale,
                      const float* k_scale, const float* v_scale, void* o, float* lse, int B,
                      int Hq, int Hkv, int Sq, int Sk, int d, int causal, float scale,
                      void* stream);

/*
 * Bytes of device workspace fa_bwd / fa_bwd_varlen need: an fp32 dQ
 * accumulator [T][Hq][d] (used by the one-pass form only), the fp32 row terms
 * -D_i = -sum_c dO_ic O_ic and -LSE*log2(e) ([Hq][P] each, P = T padded per
 * sequence), and room for two boundary lists of B+1 ints (fa_bwd_varlen copies
 * its query and key boundaries there, back to back), each region rounded up to
 * 256 bytes; T = B*Sq (dense) or total_q (packed, pass the packed row count;
 * 0 = dense).
 */
FA_API size_t fa_bwd_workspace_bytes(int B, int Hq, int Sq, int d, int total_q);

/*
 * Backward: dq, dk, dv (bf16) from q, k, v, o, lse (as written by fa_fwd) and
 * dout. dk/dv of a KV head are summed over the query heads of its group.
 * Head dim 64, 128, 192 or 256. With 192 the passes step over 64 query rows /
 * 64 keys instead of 128; with 256 each dK/dV unit accumulates one 128-column
 * half of dV and dK (S^T and dP^T recomputed per half) and the dQ pass steps
 * over 32 keys.
 * Runs three kernels on `stream`: a preprocess (the row terms -D and
 * -LSE*log2e), a dK/dV pass over key blocks and a dQ pass over query blocks.
 * Every output element is written by one CTA with a fixed summation order (no
 * atomics), so results are bitwise reproducible. `workspace` (device, 256-byte
 * aligned, >= fa_bwd_workspace_bytes) is scratch owned by the caller; its
 * contents on entry do not matter. (The one-pass form selectable with
 * fa_debug_set("bwd_mode", 0) accumulates dQ with fp32 atomics instead, so its
 * dq may differ in the last bits between runs.)
 */
FA_API int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq,
           int Sk, int d, int causal, float scale, const int* cu_seqlens, void* workspace,
           size_t workspace_bytes, void* stream);

/*
 * Backward without a caller workspace, for callers that cannot allocate
 * device memory (e.g. a runtime whose memory is all owned by its own pool
 * allocator, or a latency-critical path where cudaMalloc, which can
 * synchronise the device, is not allowed). Same arguments and results as
 * fa_bwd minus the workspace: the scratch is a fixed array of
 * FA_BWD_NOALLOC_SCRATCH_BYTES inside the library (held on every GPU that
 * loads the library until exit). Problems needing more scratch than that
 * (fa_bwd_workspace_bytes) are rejected with FA_ERR_WORKSPACE before any
 * work. The first call on a device looks up the array's device address (make
 * it before any stream capture). All calls share the array: calls that
 * overlap on the GPU race and must be serialised by the caller. Allocates no
 * memory. The FlashAttention-4 pages have no counterpart of this entry point.
 */
#define FA_BWD_NOALLOC_SCRATCH_BYTES (32u << 20)
FA_API int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                          const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                          int Hq, int Hkv, int Sq, int Sk, int d, int causal, float scale,
                          const int* cu_seqlens, void* stream);

/*
 * Packed variable-length attention with separate query and key boundaries
 * (e.g. prefill over cached keys: a sequence may have more keys than
 * queries, or fewer). Sequence i's queries are rows [cu_seqlens_q[i],
 * cu_seqlens_q[i+1]) of q/o/dout/dq ([Tq,Hq,d]) and its keys rows
 * [cu_seqlens_k[i], cu_seqlens_k[i+1]) of k/v/dk/dv ([Tk,Hkv,d]); causal masking
 * is bottom-right aligned per sequence (key j visible to query i iff
 * j <= i + k_len - q_len), as in the dense Sq != Sk case. LSE is [Hq,Tq]. Both
 * lists are device int32 arrays of nseq+1 non-decreasing entries from 0 to
 * Tq / Tk. Same method and errors as fa_fwd / fa_bwd (the pages' "variable
 * sequence lengths": "FlashAttention-4: Algorithm and Kernel Pipelining
 * Co-Design for Asymmetric Hardware Scaling", Summary); fa_bwd_varlen's
 * workspace is fa_bwd_workspace_bytes(nseq, Hq, Tq, d, Tq) bytes.
 */
FA_API int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                         int nseq, int Hq, int Hkv, int Tq, int Tk, int d, int causal, float scale,
                         const int* cu_seqlens_q, const int* cu_seqlens_k, void* stream);
FA_API int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dout, void* dq, void* dk, void* dv,
                         int nseq, int Hq, int Hkv, int Tq, int Tk, int d, int causal, float scale,
                         const int* cu_seqlens_q, const int* cu_seqlens_k, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * Combine step of context parallelism (K/V split into disjoint shards, each
 * shard's forward run separately): given, for the same queries, part p's O_p
 * and LSE_p from fa_fwd over key set p, writes the attention over the union
 * of the key sets,
 *     LSE = log sum_p exp(LSE_p),   O = sum_p exp(LSE_p - LSE) O_p
 * (the online-softmax rescale applied across parts: "FlashAttention-4
 * Conquers Asymmetric GPU Hardware Scaling", episode description, tiling with
 * an online softmax; its source list names Ring Attention, blockwise
 * attention across devices). A row that saw no key in a part (LSE = +inf,
 * O = 0, the forward's convention) counts zero; a row with no key in any part
 * gets O = 0, LSE = +inf.
 *   o_parts   device bf16, P consecutive arrays in fa_fwd's O layout
 *             ([B,S,Hq,d] dense, [S,Hq,d] packed with S = T)
 *   lse_parts device fp32, P consecutive arrays in fa_fwd's LSE layout
 *             ([B,Hq,S] dense, [Hq,T] packed)
 *   packed    0 dense, 1 packed (B is then unused)
 *   o, lse    outputs in the same layouts (must not alias the parts)
 * 1 <= P <= 64, d in {64, 128, 192, 256}; o_parts and o 16-byte aligned.
 * Asynchronous on `stream`; allocates nothing. Errors: FA_ERR_INVALID_ARG
 * (NULL or misaligned pointer, P or sizes out of range), FA_ERR_UNSUPPORTED
 * (d), FA_ERR_CUDA.
 */
FA_API int fa_merge(const void* o_parts, const float* lse_parts, int P, int B, int Hq, int S,
                    int d, int packed, void* o, float* lse, void* stream);

/*
 * Accumulation of partial gradients in fp32: acc[i] += x[i] for i < n, acc
 * fp32, x bf16 (e.g. the dQ, dK, dV that fa_bwd returns for each key shard of
 * a context-parallel backward; the gradient is their sum, the cross-shard
 * counterpart of the backward's own accumulation over key blocks:
 * "FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for Asymmetric
 * Hardware Scaling", abstract item 3). Device pointers, 16-byte aligned; n a
 * multiple of 8. Asynchronous on `stream`; allocates nothing. Errors:
 * FA_ERR_INVALID_ARG (NULL or misaligned pointer, bad n), FA_ERR_CUDA.
 */
FA_API int fa_accumulate(float* acc, const void* x, long long n, void* stream);

/*
 * out[i] = bf16(in[i]) (round to nearest even) for i < n: the final step of an
 * fp32 gradient accumulation. Same conventions and errors as fa_accumulate.
 */
FA_API int fa_to_bf16(void* out, const float* in, long long n, void* stream);

/* Static text for a status code. */
FA_API const char* fa_status_string(int status);

/* Thread-local detail of the last failing call on this thread ("" if none). */
FA_API const char* fa_last_error(void);

/*
 * Reads (and optionally clears) the current device's error word, which a
 * kernel sets when one of its bounded waits expires (the kernel then returns
 * early instead of hanging; its outputs are invalid). Synchronises the device.
 * *code receives 0 if no wait expired, else the site of the first expiry.
 * Returns FA_OK, or FA_ERR_CUDA if the read failed.
 */
FA_API int fa_get_device_error(int* code, int clear);

/*
 * Test and tuning knobs (not part of the numerical contract). Keys:
 *   "tau"        conditional-rescale threshold, base-2 units (default 0)
 *   "fp8_tau"    the same for the FP8 forward, in [0, 1.5] (default 1.5: the
 *                stored weights 2^(7 + tau) * p stay below e4m3's 448)
 *   "poly8"      forward: eighths of the exponentials computed by the FMA-pipe
 *                polynomial instead of MUFU ex2 (0, 2 or 4)
 *   "bwd_poly8"  the same for the backward
 *   "fp8_poly8"  the same for the FP8 forward
 *   "timeout_ms" bounded-wait deadline in milliseconds (default 2000)
 *   "grid"       persistent grid size override (0 = one CTA per SM)
 *   "bwd_mode"   backward form: 1 two passes (default), 2 the same with the
 *                dK/dV pass on CTA pairs (cta_group::2, head dim 128), 0 one
 *                pass with fp32 dQ atomics and a convert pass (head dim 128)
 *   "fwd_hblock" forward heads per scheduler group (0 = all heads, default)
 *   "fwd_split_q" bf16 forward (head dim <= 128): 1 loads each of a unit's two
 *                Q tiles on its own barrier pair (tile 0's next Q as soon as
 *                tile 0's last S is done), 0 both on one pair, -1 automatic
 *                (default: 1 for dense layouts with at most 4096 keys). Results
 *                are bit-identical either way.
 *   "bwd_hblock" dK/dV pass: KV heads per scheduler group (0 = automatic)
 *   "bwd_hblock_q" dQ pass: query heads per scheduler group (0 = automatic)
 *   "bwd_pdl"    two-pass backward: 1 launches the dQ pass as a programmatic
 *                dependent of the dK/dV pass, so that its CTAs start on the
 *                SMs the dK/dV pass leaves (the passes share no data; the call
 *                still completes only when both have); 0 launches it the
 *                ordinary way; -1 automatic (default: 1 for dense layouts with
 *                at most 4096 keys). Results are bit-identical.
 * Returns FA_OK or FA_ERR_INVALID_ARG. Process-wide; not thread-safe with
 * concurrent launches.
 */
FA_API int fa_debug_set(const char* key, double value);

/*
 * Measurement hook: the next fa_fwd call records `start` on its stream right
 * before its kernel and `stop` right after; the next fa_bwd call does the same
 * around its main kernel (not the preprocess/convert passes). Each event pair
 * is used once and then forgotten. Arguments are cudaEvent_t handles created by
 * the caller on the current device (NULL clears). Process-wide, like the knobs.
 */
FA_API int fa_debug_set_events(int which /* 0 = forward, 1 = backward */, void* start,
                               void* stop);

/*
 * Tuning hook: while armed, each fa_bwd main kernel writes a role timeline of
 * CTA 0 (clock64 after each cross-role wait, for its first 512 steps, and at
 * the dK/dV pass's unit boundaries) into trace_dev (device buffer of at least
 * 26*512 int64). NULL disarms. Errors: FA_ERR_INVALID_ARG (buffer too small).
 */
FA_API int fa_debug_set_trace(void* trace_dev, size_t bytes);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
