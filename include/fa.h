/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact attention forward library (libfa.so).
 *
 * The operation (all entry points): for every batch b, head h and query row i,
 *
 *     O[b,h,i,:] = sum_j softmax_j( scale * q_i . k_j  + mask(i,j) ) * v_j
 *     LSE[b,h,i] = ln sum_{j allowed} exp(scale * q_i . k_j)
 *
 * with mask(i,j) = -inf when causal and j > i + (Nk - Nq) (the diagonal is
 * aligned to the bottom-right corner, which is the usual "row i sees j <= i"
 * when Nq == Nk), else 0.  The computation follows the FlashAttention-2
 * forward: Q row-blocks outer, K/V tiles inner, a running row max m and row
 * sum l, the output rescaled by exp(m_old - m_new) and divided by l once at the
 * end, and LSE = m + ln l written per row.  Sources: "6.2 FlashAttention V2
 * explained" §3.2 (deferred rescaling), §5 (causal mask and block skipping),
 * §6 (the forward algorithm with its L = m + log l output); "02 · FA2:
 * parallelism and work partitioning" §2 (a grid over Q row-blocks, and for
 * seqlen_q = 1 the split-KV partials (O, LSE) merged by a combine kernel).
 *
 * Layouts: q, o are [B, H, Nq, d]; k, v are [B, H, Nk, d]; all contiguous
 * (row stride d elements), 16-bit (fp16 or bf16, the same for all four).
 * lse is [B, H, Nq] fp32.  Accumulation is fp32.
 *
 * Ownership: the caller owns every buffer and the stream.  All pointers are
 * device pointers unless stated otherwise.  The library allocates no device
 * memory; it keeps only a per-device status word for device-side errors.
 *
 * Asynchrony: every launching call is asynchronous on `stream`.  Its return
 * value reports host-side validation and launch errors only; errors raised on
 * the device (a bounded wait that ran out) are reported by
 * fa_get_device_status.
 *
 * Common validation (returned before anything is launched):
 *   FA_ERR_INVALID_ARG   B, H, Nq, Nk <= 0; scale not finite or <= 0; a null
 *                        q, k, v or o; an unknown dtype; causal not 0/1.
 *   FA_ERR_UNSUPPORTED   d not 64 or 128.
 *   FA_ERR_MISALIGNED    q, k, v, o not 16-byte aligned (TMA requirement),
 *                        lse not 4-byte aligned.
 *   FA_ERR_CUDA          a CUDA runtime error at launch.
 * Inputs q, k, v are never written; o and lse are fully overwritten.  A row
 * that sees no key (only possible when causal and Nq > Nk) gets O = 0 and
 * LSE = -inf.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *fa_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum { FA_F16 = 0, FA_BF16 = 1 } fa_dtype;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = -1,
    FA_ERR_UNSUPPORTED = -2,
    FA_ERR_MISALIGNED = -3,
    FA_ERR_WORKSPACE = -4,
    FA_ERR_CUDA = -5,
    FA_ERR_DEVICE_TIMEOUT = -6,
    FA_ERR_SCRATCH_LIMIT = -7
} fa_status;

/*
 * Fused attention forward (one launch): one CTA per 128 query rows and head,
 * K/V tiles streamed by TMA, both GEMMs on tcgen05 tensor cores with fp32
 * accumulators in tensor memory, online softmax with deferred 1/l.  Under
 * causal masking, K/V tiles entirely above the diagonal are skipped and only
 * tiles that straddle it (or the ragged Nk tail) are masked element-wise.
 * ("6.2 FlashAttention V2 explained" §6; "02 · FA2" §2 and §4.)
 *
 *   q, k, v  inputs, layouts above.
 *   o        output [B, H, Nq, d], same dtype as the inputs.
 *   lse      output [B, H, Nq] fp32 (natural log of the scaled scores), or NULL.
 *   scale    score scale, normally 1/sqrt(d).
 * Returns FA_OK or one of the validation errors above, or FA_ERR_INVALID_ARG
 * when B*H > 65535 (one grid dimension per head).
 */
FA_API int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
           int B, int H, int Nq, int Nk, int d, int causal, float scale,
           fa_dtype dtype, fa_stream_t stream);

/*
 * Workspace bytes that fa_fwd_splitkv needs for `num_splits` splits:
 * fp32 partial outputs [num_splits, B, H, Nq, d] followed by fp32 partial LSEs
 * [num_splits, B, H, Nq], each region 256-byte aligned.  num_splits <= 0 means
 * the value fa_splitkv_num_splits would choose.  Returns 0 on invalid sizes.
 */
FA_API size_t fa_splitkv_workspace_bytes(int B, int H, int Nq, int Nk, int d, int num_splits);

/*
 * The number of splits fa_fwd_splitkv uses when passed num_splits <= 0
 * (enough CTAs to fill the GPU several times over, at most 64), and the key
 * count of every split but the last: split s covers keys
 * [s * split_len, min((s + 1) * split_len, Nk)), where split_len is a multiple
 * of the 64-key tile.  A split may be empty when num_splits exceeds the tile count.
 */
FA_API int fa_splitkv_num_splits(int B, int H, int Nq, int Nk, int d);
FA_API int fa_splitkv_split_len(int Nk, int num_splits);

/*
 * Split-KV attention forward (flash-decoding), written for Nq = 1 but valid for
 * any Nq: the keys of each (b, h) are cut into num_splits contiguous ranges;
 * one CTA per (split, query row, head) computes the range's normalised partial
 * output O_s and LSE_s on CUDA cores (fp32), then a combine kernel merges them
 * ("02 · FA2: parallelism and work partitioning" §2, decode / split-KV).
 * Two launches on `stream`; the partials live in the caller's workspace.
 *
 *   num_splits       1..256, or <= 0 for fa_splitkv_num_splits.
 *   workspace        device buffer of at least
 *                    fa_splitkv_workspace_bytes(B, H, Nq, Nk, d, num_splits)
 *                    bytes, 256-byte aligned; its contents are overwritten.
 * Errors: the common ones, plus FA_ERR_WORKSPACE when the workspace is NULL,
 * misaligned or too small, and FA_ERR_INVALID_ARG when num_splits > 256.
 */
FA_API int fa_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                   int B, int H, int Nq, int Nk, int d, int causal, float scale,
                   fa_dtype dtype, int num_splits, void *workspace, size_t workspace_bytes,
                   fa_stream_t stream);

/*
 * Grouped-query attention (GQA; multi-query attention when H_kv = 1): H query
 * heads share H_kv K/V heads, `H / H_kv` consecutive query heads per K/V head,
 * so query head h of batch entry b reads K/V head h / (H / H_kv) of that entry:
 *
 *     O[b,h,i,:] = sum_j softmax_j( scale * q[b,h,i] . k[b,h/g,j] + mask ) v[b,h/g,j],  g = H / H_kv
 *
 * Otherwise these are fa_fwd and fa_fwd_splitkv (which are the case H_kv = H):
 * q, o are [B, H, Nq, d]; k, v are [B, H_kv, Nk, d]; lse is [B, H, Nq]; the
 * split-KV workspace is sized by fa_splitkv_workspace_bytes(B, H, ...) as for
 * multi-head attention.  ("Flash Attention (4)" §5: the K/V index mapped per
 * group of query heads; "Lecture 25" §0.3, its table's GQA entry.)
 * fa_fwd_gqa without causal masking, or with Nq = 1 (decode, where the one
 * query row sees every key), treats the H/H_kv query heads of a K/V head as
 * one head of (H/H_kv)*Nq query rows: q, o and lse hold them consecutively, so
 * the group's rows share each K/V tile on the tensor cores and K/V is read
 * once per group.
 * Errors: as fa_fwd / fa_fwd_splitkv, plus FA_ERR_INVALID_ARG when H_kv <= 0
 * or H is not a multiple of H_kv.
 */
/*
 * Variable-length batch (packed sequences): num_seqs sequences of different
 * lengths in one launch, each attending only within itself.  q, o are packed
 * [total_q, H, d] and k, v [total_k, H_kv, d] (token-major, contiguous, 16-bit);
 * lse is [H, total_q] fp32 or NULL.  cu_seqlens_q and cu_seqlens_k are DEVICE
 * arrays of num_seqs + 1 int32 offsets: sequence s owns query tokens
 * [cu_seqlens_q[s], cu_seqlens_q[s+1]) and keys [cu_seqlens_k[s], cu_seqlens_k[s+1]).
 * Per sequence this is fa_fwd_gqa with Nq = its query length, Nk = its key
 * length (the causal diagonal aligned to its bottom-right corner); a sequence
 * with no key gets O = 0 and LSE = -inf.  The caller guarantees
 * 0 = cu[0] <= cu[1] <= ... <= cu[num_seqs] = total for both arrays and that no
 * sequence has more than max_seqlen_q query tokens (the grid is sized by it);
 * the offsets are read on the device only.  A key tile may extend past its
 * sequence into the next one; those keys get weight exactly 0, so K and V must
 * be finite everywhere (0 * inf is NaN).  ("Flash Attention (4)" §5: an entry
 * with cu_seqlens; "Lecture 25" §7.1 item 07 and §7.2 item 2: sequence packing
 * without padding.)
 * Errors: the common ones (with total_q, total_k in the places of Nq, Nk), and
 * FA_ERR_INVALID_ARG for null offsets, num_seqs <= 0, max_seqlen_q outside
 * [1, total_q], H not a multiple of H_kv, or num_seqs * H > 65535;
 * FA_ERR_MISALIGNED for offsets not 4-byte aligned.
 */
FA_API int fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
           const int *cu_seqlens_q, const int *cu_seqlens_k, int num_seqs, int max_seqlen_q,
           int total_q, int total_k, int H, int H_kv, int d, int causal, float scale,
           fa_dtype dtype, fa_stream_t stream);
/*
 * The same variable-length forward launched over a work list instead of a
 * (max_seqlen_q / 128) x (num_seqs * H) grid: a first launch on `stream` reads
 * cu_seqlens_q on the device and writes into `workspace` the (sequence, row
 * block) pairs that hold rows, longest sequences first and each sequence's
 * heaviest causal row block first; the forward then runs one CTA per pair and
 * head, so no CTA is spent on row blocks past a sequence's end and no
 * max_seqlen_q is needed.  Results are bit for bit those of fa_fwd_varlen.
 * ("02 · FA2" §2: the sequence dimension as a unit of parallel work; "Lecture
 * 25" §7.2 item 2: packing without padding.)
 * Workspace: device memory of at least fa_fwd_varlen_workspace_bytes(num_seqs,
 * total_q) = 16 + 8 * (ceil(total_q / 128) + num_seqs) bytes, 16-byte aligned,
 * owned by the caller and free for reuse once the call's work on `stream` has
 * finished.  The work list is built by one CTA in num_seqs^2 / 1024 steps per
 * thread, small next to the attention itself for any practical batch.
 * Errors: as fa_fwd_varlen (without the max_seqlen_q checks; H > 65535 is
 * FA_ERR_INVALID_ARG), and FA_ERR_WORKSPACE for a null, misaligned or short
 * workspace.
 */
FA_API size_t fa_fwd_varlen_workspace_bytes(int num_seqs, int total_q);
FA_API int fa_fwd_varlen_ws(const void *q, const void *k, const void *v, void *o, float *lse,
                            const int *cu_seqlens_q, const int *cu_seqlens_k, int num_seqs, int total_q,
                            int total_k, int H, int H_kv, int d, int causal, float scale, fa_dtype dtype,
                            void *workspace, size_t workspace_bytes, fa_stream_t stream);

FA_API int fa_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse,
           int B, int H, int H_kv, int Nq, int Nk, int d, int causal, float scale,
           fa_dtype dtype, fa_stream_t stream);
FA_API int fa_fwd_splitkv_gqa(const void *q, const void *k, const void *v, void *o, float *lse,
                   int B, int H, int H_kv, int Nq, int Nk, int d, int causal, float scale,
                   fa_dtype dtype, int num_splits, void *workspace, size_t workspace_bytes,
                   fa_stream_t stream);

/*
 * LSE-weighted merge of split partials, per row r of B*H*Nq rows:
 *   M = max_s LSE_s;  w_s = exp(LSE_s - M);
 *   O = sum_s w_s O_s / sum_s w_s;  LSE = M + ln sum_s w_s.
 * A row whose partials are all empty (every LSE_s = -inf) gets O = 0, LSE = -inf.
 *
 *   o_part    fp32 [num_splits, B, H, Nq, d], normalised partial outputs.
 *   lse_part  fp32 [num_splits, B, H, Nq].
 *   o         [B, H, Nq, d] in `dtype`;  lse  [B, H, Nq] fp32 or NULL.
 * Errors: FA_ERR_INVALID_ARG (sizes, null pointers, num_splits not in 1..256),
 * FA_ERR_UNSUPPORTED (d), FA_ERR_MISALIGNED (o_part, o not 16-byte aligned).
 */
FA_API int fa_splitkv_combine(const float *o_part, const float *lse_part, void *o, float *lse,
                       int num_splits, int B, int H, int Nq, int d, fa_dtype dtype,
                       fa_stream_t stream);

/*
 * Split-KV attention forward that allocates nothing and needs no workspace.
 * (No counterpart in the source pages: this is a library convenience.)
 *
 * For callers that cannot allocate device memory at the point of the call --
 * code running inside a CUDA graph capture or a memory-pool-less runtime, a
 * host that must not grow its footprint after start-up, a caller without a
 * device allocator of its own -- this variant keeps the split partials in a
 * fixed scratch array built into the library (a file-scope __device__ array of
 * fa_splitkv_noalloc_capacity_bytes() = 16 MiB, held on every GPU that loads
 * the library until the process exits).  It calls no cudaMalloc or cudaFree.
 *
 * Arguments and results are those of fa_fwd_splitkv without the workspace;
 * the caller still provides q, k, v, o and lse.  The partials need
 * num_splits * B * H * Nq * (d + 1) * 4 bytes (each of the two regions rounded
 * up to 256 bytes); a problem that does not fit returns FA_ERR_SCRATCH_LIMIT
 * before anything is launched (use fewer splits, or fa_fwd_splitkv).
 *
 * The first call on a device looks up the scratch array's device address with
 * that device current; make that first call before any stream capture.  All
 * calls in the process share the one array and every call overwrites it, so
 * two calls whose kernels overlap on the GPU (different streams without
 * ordering between them) race and give wrong results.  Nothing in the scratch
 * needs clearing: every partial is written before the combine reads it.
 */
FA_API int fa_fwd_splitkv_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                                  int B, int H, int Nq, int Nk, int d, int causal, float scale,
                                  fa_dtype dtype, int num_splits, fa_stream_t stream);

/* Bytes of the built-in scratch used by fa_fwd_splitkv_noalloc (16 MiB). */
FA_API size_t fa_splitkv_noalloc_capacity_bytes(void);

/*
 * Forward from and to HOST memory, with the copies overlapped with the compute.
 * q_host, k_host, v_host, o_host, lse_host hold what fa_fwd_gqa's q, k, v, o, lse
 * hold, in the same layouts, in host memory (lse_host may be NULL).  The K/V
 * heads (B * H_kv of them, with their H / H_kv query heads each) are cut into
 * num_chunks consecutive chunks (num_chunks <= 0: min(B * H_kv, 8)); chunk c's
 * inputs are copied to the device on a copy stream while chunk c - 1 is computed
 * on `stream` and chunk c - 2's output is copied back on a second copy stream.
 * Each chunk runs the fa_fwd_gqa kernels on its heads, so o and lse equal
 * fa_fwd_gqa's bit for bit.  The call is ordered on `stream` like a kernel
 * launch: the copies start after the work queued on `stream` before the call,
 * and o_host, lse_host hold the result once `stream` has reached the point of the
 * call's return (synchronize `stream` before reading them).  Host buffers should
 * be page-locked (cudaHostAlloc / cudaHostRegister); with pageable memory the
 * results are the same but the copies do not overlap.
 * Workspace: device memory of at least fa_fwd_host_workspace_bytes(B, H, H_kv,
 * Nq, Nk, d) bytes, 256-byte aligned, owned by the caller (the device copies of
 * q, k, v, o and lse); free for reuse once `stream` has passed the call.  The
 * two copy streams and their events belong to the library (one set per device;
 * concurrent calls on one device share them, which orders their copies).
 * Errors: as fa_fwd_gqa; FA_ERR_INVALID_ARG for a null host pointer (lse_host
 * excepted); FA_ERR_WORKSPACE for a null, misaligned or short workspace;
 * FA_ERR_CUDA if a copy or stream operation fails (outputs then unspecified).
 * (The pages time the kernel with its inputs resident; this entry point is the
 * end-to-end form of the same "Flash Attention (4)" §5 forward.)
 */
FA_API size_t fa_fwd_host_workspace_bytes(int B, int H, int H_kv, int Nq, int Nk, int d);
FA_API int fa_fwd_host(const void *q_host, const void *k_host, const void *v_host, void *o_host, float *lse_host,
                       int B, int H, int H_kv, int Nq, int Nk, int d, int causal, float scale, fa_dtype dtype,
                       int num_chunks, void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Attention backward: the gradients dQ, dK, dV of O = softmax(scale * Q K^T +
 * mask) V given dO, for the same mask as the forward ("Lecture 25" §3.3, the
 * backward with P recomputed from the saved statistics; "02 · FA2:
 * parallelism and work partitioning" §5, the K/V block outer loop with dQ
 * accumulated across blocks):
 *     P = exp(scale * Q K^T + mask - LSE),  dV = P^T dO,  dP = dO V^T,
 *     dS = P o (dP - rowsum(dO o O)),  dQ = scale * dS K,  dK = scale * dS^T Q.
 * Inputs: q, k, v, dtype and causal as given to the forward that produced o
 * and lse (lse in natural-log units, as fa_fwd writes it; a row with LSE = -inf
 * gets dQ = 0); dout is dO.  Layouts: q, o, dout, dq [B, H, Nq, d]; k, v, dk, dv
 * [B, H, Nk, d]; lse [B, H, Nq] fp32; 16-bit tensors contiguous.  Outputs dq,
 * dk, dv are fully overwritten (keys that no query sees get dK = dV = 0).
 * Workspace: device memory of at least fa_bwd_workspace_bytes(B, H, Nq, d)
 * bytes, 256-byte aligned, owned by the caller and free for reuse once the
 * call's work on `stream` has finished; it holds an fp32 dQ accumulator and
 * two per-row vectors.  The dQ sum over K/V blocks uses fp32 atomic adds, so
 * dq may differ in the last bits between runs; dk and dv are deterministic.
 * Three launches on `stream`: preprocess, the main kernel, dQ conversion.
 * Errors: the common validation above; FA_ERR_INVALID_ARG for a null dout,
 * lse, dq, dk or dv, or B * H > 65535; FA_ERR_MISALIGNED for dout, dq, dk, dv
 * not 16-byte aligned; FA_ERR_WORKSPACE for a null, misaligned or short
 * workspace.
 */
FA_API size_t fa_bwd_workspace_bytes(int B, int H, int Nq, int d);
/* Grouped-query form: k, v, dk, dv are [B, H_kv, Nk, d] with H_kv dividing H (query
 * head h reads K/V head h / (H / H_kv), as in fa_fwd_gqa); a K/V head's dK and dV
 * sum the contributions of the H / H_kv query heads that read it.  fa_bwd is the
 * case H_kv = H.  FA_ERR_INVALID_ARG if H_kv does not divide H. */
FA_API int fa_bwd_gqa(const void *q, const void *k, const void *v, const void *o, const void *dout,
                      const float *lse, void *dq, void *dk, void *dv, int B, int H, int H_kv, int Nq, int Nk, int d,
                      int causal, float scale, fa_dtype dtype, void *workspace, size_t workspace_bytes,
                      fa_stream_t stream);
FA_API int fa_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout, const float *lse,
                  void *dq, void *dk, void *dv, int B, int H, int Nq, int Nk, int d, int causal, float scale,
                  fa_dtype dtype, void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Backward of a variable-length (packed) batch: the gradients of fa_fwd_varlen,
 * sequence by sequence the gradients of fa_bwd_gqa with Nq, Nk the sequence's
 * lengths.  Layouts as in fa_fwd_varlen: q, o, dout, dq packed [total_q, H, d];
 * k, v, dk, dv [total_k, H_kv, d]; lse [H, total_q] fp32 as fa_fwd_varlen wrote
 * it; cu_seqlens_q, cu_seqlens_k DEVICE arrays of num_seqs + 1 int32 offsets with
 * the same guarantees as there.  max_seqlen_k must lie in [1, total_k] (it is
 * checked but no longer sizes the grid: the CTAs follow a work list of the
 * (sequence, key block) pairs that hold keys, built on the device from
 * cu_seqlens_k, longest sequences first and each sequence's key blocks in
 * ascending order, the causal heaviest first).  Every query token's dq and every
 * key token's dk, dv are written;
 * a sequence without query tokens gets dK = dV = 0, one without keys dQ = 0.
 * Q, K, V and dO must be finite everywhere: a tile may read tokens of the
 * neighbouring sequence and weights them by exactly 0.
 * Workspace: at least fa_bwd_varlen_workspace_bytes(num_seqs, total_q, total_k,
 * H, d) bytes, 256-byte aligned, owned by the caller; besides the buffers of
 * fa_bwd it holds each sequence's first row in a per-head row space where
 * sequences start on multiples of 128 rows, computed on the device from
 * cu_seqlens_q, and the work list (16 + 8 * (ceil(total_k / 128) + num_seqs)
 * bytes).  Five launches on `stream` (the two plans, then those of fa_bwd).
 * ("Flash Attention (4)" §5: the entry with cu_seqlens; "Lecture 25" §3.3: the
 * recomputing backward.)
 * Errors: the common validation (total_q, total_k in the places of Nq, Nk);
 * FA_ERR_INVALID_ARG for a null dout, lse, dq, dk, dv or offset array,
 * num_seqs <= 0, max_seqlen_k outside [1, total_k], H not a multiple of H_kv,
 * or H_kv > 65535; FA_ERR_MISALIGNED for dout, dq, dk, dv not 16-byte
 * or offsets not 4-byte aligned; FA_ERR_WORKSPACE for a null, misaligned or
 * short workspace.
 */
FA_API size_t fa_bwd_varlen_workspace_bytes(int num_seqs, int total_q, int total_k, int H, int d);
FA_API int fa_bwd_varlen(const void *q, const void *k, const void *v, const void *o, const void *dout,
                         const float *lse, void *dq, void *dk, void *dv, const int *cu_seqlens_q,
                         const int *cu_seqlens_k, int num_seqs, int max_seqlen_k, int total_q, int total_k, int H,
                         int H_kv, int d, int causal, float scale, fa_dtype dtype, void *workspace,
                         size_t workspace_bytes, fa_stream_t stream);

/*
 * FP8 (E4M3) forward with per-block scales ("Flash Attention (4)" §5.4: both
 * products in E4M3, block-wise scale factors against underflow).
 *
 * fa_fp8_quantize: x [BH, N, d] 16-bit (dtype) to E4M3 codes, one fp32 scale per
 * block of 128 rows of one head: s = amax / 448 (1 for an all-zero block) and
 * code = E4M3(x / s) (fp32 division; round to nearest, ties to even; magnitudes
 * above 448 saturate).  scales is [BH, ceil(N/128)].  transpose = 0 writes x8 as
 * [BH, N, d] (the layout of q8 and k8); transpose = 1 writes it as
 * [BH, d, ceil(N/128)*128] with zero codes past N (the layout of v8t).
 *
 * fa_fwd_fp8: O and LSE of attention over the dequantized inputs (Q = q8 x
 * q_scale of each 128-row block, likewise K and V), causal as fa_fwd.  q8, k8:
 * [B, H, Nq or Nk, d] codes; v8t: [B, H, d, ceil(Nk/128)*128] codes; q_scale
 * [B*H, ceil(Nq/128)], k_scale and v_scale [B*H, ceil(Nk/128)]; o [B, H, Nq, d] in
 * out_dtype; lse [B, H, Nq] fp32 or NULL.  Both products run in E4M3 with fp32
 * accumulation; P is rounded to E4M3 after scaling by 2^7 times the V block's scale
 * over the head's largest V scale, so its relative rounding error is at most 2^-4
 * (absolute 2^-10 / that factor below 2^-6).  d must be 128 (FA_ERR_UNSUPPORTED
 * otherwise).  Errors: FA_ERR_INVALID_ARG for null pointers, non-positive sizes,
 * B*H > 65535, a bad scale or dtype; FA_ERR_MISALIGNED for code tensors or o not
 * 16-byte aligned, scales or lse not 4-byte aligned.
 */
FA_API int fa_fp8_quantize(const void *x, void *x8, float *scales, int BH, int N, int d, int transpose,
                           fa_dtype dtype, fa_stream_t stream);
FA_API int fa_fwd_fp8(const void *q8, const float *q_scale, const void *k8, const float *k_scale, const void *v8t,
                      const float *v_scale, void *o, float *lse, int B, int H, int Nq, int Nk, int d, int causal,
                      float scale, fa_dtype out_dtype, fa_stream_t stream);

/*
 * Self-test of device-side failure reporting: launches one warp that waits on an
 * mbarrier nothing will complete, gives up after limit_ms (1..10000) exactly as
 * the attention kernels' bounded waits do, and sets the device status word; the
 * next fa_get_device_status on that stream returns FA_ERR_DEVICE_TIMEOUT and
 * clears it.  Nothing faults, traps or hangs; the context stays usable.
 */
FA_API int fa_selftest_timeout(int limit_ms, fa_stream_t stream);

/*
 * The reason for the last FA_ERR_CUDA returned to the calling thread (the CUDA
 * call that failed and its error name), or "" if there was none.  The string
 * belongs to the library and stays valid until this thread's next call.
 */
FA_API const char *fa_last_error(void);

/*
 * Synchronises `stream`, then returns FA_ERR_DEVICE_TIMEOUT if any kernel of
 * this library on the current device gave up a bounded wait since the last
 * call (the flag is cleared), FA_ERR_CUDA if the context reports an error,
 * else FA_OK.
 */
FA_API int fa_get_device_status(fa_stream_t stream);

/* Static description of a status code. Never NULL. */
FA_API const char *fa_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
FA_API int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
