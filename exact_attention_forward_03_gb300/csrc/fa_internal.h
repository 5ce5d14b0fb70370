// fa_internal.h -- host-side interface between the C ABI (fa_api.cu) and the
// kernel translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

// Device-side error bits OR-ed into the per-device status word.
constexpr int kDevErrTimeout = 1;
constexpr int kDevErrLayout = 2;  // a kernel found its shared memory base misaligned

// Tile shape of the fused forward kernel: 128 query rows per Q tile (one TMEM
// lane per row), one Q tile per CTA, 128 keys per K/V tile.
constexpr int kFwdBr = 128;
constexpr int kFwdBc = 128;
constexpr int kFwdTilesPerCta = 1;
// Keys per tile of the split-KV kernel; split lengths are multiples of it.
constexpr int kDecBc = 64;
constexpr int kMaxSplits = 256;

struct FwdArgs {
    void *o;        // [BH, Nq, d] 16-bit
    float *lse;     // [BH, Nq] or nullptr
    int *status;    // device status word
    int Nq, Nk;
    int num_m;      // ceil(Nq / (kFwdTilesPerCta * kFwdBr)): row blocks per head
    int H;          // query heads per batch entry
    // Launch order: CTAs take the row blocks (list entries) of head_group heads at a
    // time, the heaviest block of each of those heads first (see fa_fwd_kernel).
    int head_group;
    int group;      // query heads per K/V head (H / H_kv)
    // Variable-length batches (packed [total, heads, d] tensors): per-sequence token
    // offsets, cu_q[s]..cu_q[s+1] and cu_k[s]..cu_k[s+1]; null for dense [B, H, N, d].
    const int *cu_q;
    const int *cu_k;
    int total_q;    // tokens in the packed q (the lse layout is [H, total_q])
    // Planned variable-length launches: work[0] = number of row blocks with rows, then
    // (sequence, row block) pairs from work[2] on, longest sequences first and each
    // sequence's heaviest (last) row block first; null for the unplanned grid.
    const int *work;
    int num_seqs;
    int causal;
    float scale_log2;  // scale * log2(e)
};

struct SplitArgs {
    const void *q;     // [BH, Nq, d] 16-bit
    float *o_part;     // [S, BH, Nq, d] fp32
    float *lse_part;   // [S, BH, Nq] fp32
    int *status;
    int Nq, Nk, BH;
    int H, group;      // query heads per batch entry; query heads per K/V head
    int num_splits, split_len;
    int causal;
    float scale_log2;
};

struct CombineArgs {
    const float *o_part;
    const float *lse_part;
    void *o;
    float *lse;
    int num_splits;
    long long rows;  // BH * Nq
};

// Backward: one CTA per 128-key block and K/V head; query blocks of 128 rows of
// every query head that reads that K/V head.
constexpr int kBwdBr = 128;
constexpr int kBwdBc = 128;

struct BwdArgs {
    const void *o;      // [BH, Nq, d] 16-bit (forward output)
    const void *dout;   // [BH, Nq, d] 16-bit
    const float *lse;   // [BH, Nq] natural-log LSE of the forward
    void *dk, *dv;      // [B * H / group, Nk, d] 16-bit (one per K/V head)
    void *dq;           // [BH, Nq, d] 16-bit
    float *dq_acc;      // [BH, Nq_pad, d] fp32 workspace (zeroed by the preprocess kernel)
    float *lse2;        // [BH, Nq_pad] -LSE * log2(e); -inf for padding and rows that see no key
    float *dvec;        // [BH, Nq_pad] -D_i = -rowsum(dO_i * O_i); 0 for padding
    int *status;
    int BH, Nq, Nk, Nq_pad;   // BH = B * H query heads
    int H, group;             // query heads per batch entry; query heads per K/V head
    int causal;
    float scale;       // softmax scale
    float scale_log2;  // scale * log2(e)
    // Variable-length batches (packed [total, heads, d] tensors; lse [H, total_q]):
    // token offsets per sequence, and row_off[s], the first row of sequence s in the
    // workspace's per-head row space, where every sequence starts on a multiple of
    // 128 rows (written by the plan kernel); rows_pad rows per head.  Null for dense.
    const int *cu_q, *cu_k;
    int *row_off;
    int num_seqs, total_q, rows_pad;
    // Work list of the main kernel's CTAs (packed batches): work[0] = number of
    // (sequence, key block) pairs with keys, the pairs from work[2] on, longest
    // sequences first and each sequence's key blocks in ascending order (key block 0
    // sees the most query blocks under the causal mask).  Null for dense.
    const int *work;
};

// FP8 (E4M3) forward: blocks of 128 rows of one head carry one fp32 scale each.
struct Fp8QuantArgs {
    const void *x;   // [BH, N, d] 16-bit, d = 128
    void *x8;        // [BH, N, d] codes, or [BH, d, ld_t] when transposed
    float *scales;   // [BH, num_blocks]
    int N, num_blocks;
    int ld_t;        // row length of the transposed output (num_blocks * 128)
};

struct Fp8FwdArgs {
    void *o;               // [BH, Nq, d] 16-bit
    float *lse;            // [BH, Nq] or nullptr
    const float *q_scale;  // [BH, num_m]
    const float *k_scale;  // [BH, ceil(Nk / 128)]
    const float *v_scale;  // [BH, ceil(Nk / 128)]
    int *status;
    int Nq, Nk, num_m, causal;
    float scale_log2;      // scale * log2(e)
};

// Each launcher returns the CUDA error of the launch (cudaSuccess when queued).
// The fused forward: `to` is O's tensor map (the same boxes as Q's), for the TMA
// stores of the epilogue.  pair (d = 64 only): the form that runs two CTAs per SM,
// each with one score buffer (see fwd_pair in the C ABI).
cudaError_t launch_fwd(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &to, const FwdArgs &a, int BH, cudaStream_t stream, bool pair = false);
// Variable-length form: grid (num_m, num_seqs * H), packed tensor maps (x = column,
// y = head, z = token), a.cu_q / a.cu_k set.
cudaError_t launch_fwd_varlen(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                              const CUtensorMap &to, const FwdArgs &a, int num_seqs, cudaStream_t stream);
// Planned form: one launch writes the work list (at most `capacity` = ceil(total_q /
// 128) + num_seqs pairs) into `work`, then the forward runs on a grid of
// (capacity, H) CTAs, CTAs past the list's end leaving at entry.
// Work list of a packed batch from the offsets `cu` (num_seqs + 1 of them): work[0] =
// the number of 128-token blocks that hold tokens, then (sequence, block) pairs,
// sequences ordered by block count (descending, ties by index), each sequence's
// blocks last-first (`last_first`) or first-first.  One CTA; at most
// ceil(total / 128) + num_seqs pairs.
cudaError_t launch_varlen_plan(const int *cu, int num_seqs, int *work, bool last_first, cudaStream_t stream);
cudaError_t launch_fwd_varlen_planned(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk,
                                     const CUtensorMap &tv, const CUtensorMap &to, const FwdArgs &a, int *work,
                                     int capacity, cudaStream_t stream);
cudaError_t launch_splitkv(int d, bool bf16, const CUtensorMap &tk, const CUtensorMap &tv, const SplitArgs &a,
                           cudaStream_t stream);
cudaError_t launch_combine(int d, bool bf16, const CombineArgs &a, cudaStream_t stream);
cudaError_t launch_fp8_quant(bool bf16, bool transpose, const Fp8QuantArgs &a, int BH, cudaStream_t stream);
cudaError_t launch_fwd_fp8(bool bf16_out, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           const Fp8FwdArgs &a, int BH, cudaStream_t stream);
// A wait on an mbarrier that never completes, given up after limit_ms.
cudaError_t launch_selftest_timeout(int *status, int limit_ms, cudaStream_t stream);
// Backward: preprocess (D, lse2, zero dq_acc), the main K/V-block kernel, dQ conversion.
cudaError_t launch_bwd(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &tdo, const BwdArgs &a, cudaStream_t stream);
// Variable-length form: packed tensor maps (column, head, token), a.cu_q, a.cu_k,
// a.row_off set, `work` a buffer of 16 + 8 * capacity bytes for the key-block work
// list (capacity = ceil(total_k / 128) + num_seqs); grid (capacity, H_kv).
cudaError_t launch_bwd_varlen(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                              const CUtensorMap &tdo, const BwdArgs &a, int *work, int capacity, cudaStream_t stream);

}  // namespace fa
