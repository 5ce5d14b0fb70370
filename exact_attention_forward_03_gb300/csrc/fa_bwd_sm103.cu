// fa_bwd_sm103.cu -- attention backward on sm_103a tensor cores.
//
// Gradients of O = softmax(scale * Q K^T + mask) V for a given dO, with P
// recomputed from the forward's LSE instead of stored ("Lecture 25" §3.3):
//   dV = P^T dO,   dP = dO V^T,   dS = P o (dP - D),   D_i = rowsum(dO_i o O_i),
//   dQ = scale * dS K,   dK = scale * dS^T Q.
// (D_i = rowsum(dP_i o P_i) because dP_i . P_i = dO_i . (P_i V) = dO_i . O_i.)
// Three launches:
//   1. preprocess: D_i, LSE_i * log2(e) (+inf for a row that sees no key and for
//      the padding rows up to a multiple of 128), and a zeroed fp32 dQ accumulator;
//   2. main: one CTA per 128-key block and K/V head keeps K_j, V_j and the dK_j,
//      dV_j accumulators on chip and walks the query blocks that see the block, of
//      every query head that reads the K/V head (grouped-query attention sums
//      those heads' contributions to dK and dV on chip)
//      ("02 · FA2: parallelism and work partitioning" §5: the K/V block fixed, the
//      Q blocks in the inner loop, dQ summed across CTAs with atomic adds);
//   3. dQ = scale * accumulator, rounded to 16 bits.
//
// Main kernel, per query block i (rows q0 = 128 i ... q0 + 127), with the
// products transposed so that tensor-memory lanes are keys:
//   S^T  = K Q_i^T        M = 128 keys, N = 128 queries, K = d   -> TMEM [0,128)
//   dP^T = V dO_i^T       the same shape                          -> TMEM [128,256)
//   P^T  = 2^(S^T scale log2(e) - LSE_i log2(e)), masked; 16-bit pairs written by
//          the thread that read the scores over the first half of its 64 columns
//   dS^T = P^T o (dP^T - D), 16-bit, to shared memory as [keys][queries]
//   dV  += P^T dO_i       A = P^T from TMEM, B = dO_i MN-major    -> TMEM dV
//   dK  += dS^T Q_i       A = dS^T K-major, B = Q_i MN-major      -> TMEM dK
//   d=128: dQ_i^T = K^T dS^T  (A = K MN-major, B = dS^T MN-major) -> TMEM [128,256)
//   d=64:  dQ_i   = dS K      (A = dS MN-major, B = K MN-major)   -> TMEM [384,448)
// Every shared-memory tile is [rows][d] (or [keys][queries] for dS^T) in 64-column
// blocks of 128-byte swizzled rows, which the tensor core reads K-major in the
// first two products and MN-major in the last ones: no tile is stored twice.
//
// Roles (16 warps, four warpgroups):
//   warps 0-7   elementwise: warp w works on key lanes 32 (w % 4) ... + 31 and query
//               columns 64 (w / 4) ... + 63 (P, then dS), then the dK, dV epilogue
//   warps 8-11  dQ writers: read dQ(t) out of tensor memory (for d = 128 the lanes
//               of dQ^T are head-dim indices, so a warp's atomic adds cover 32
//               consecutive floats of a dQ row) and add it to the fp32 accumulator
//   warp 12     TMA: K_j and V_j once; Q_t with its LSE and D vectors, and dO_t,
//               through two-slot rings
//   warp 13     owns tensor memory; one lane issues every MMA
//
// Order on the tensor core per block t: dP(t), dV(t), S(t+1), dK(t), dQ(t).  S(t+1)
// overwrites P(t) once dV(t) completed and runs ahead of dK(t) and dQ(t), so the
// elementwise warps compute P(t+1) while the tensor core finishes block t; P(t)
// overlaps dP(t) and dS(t) overlaps dV(t).  For d = 128, dQ^T(t) lives in the
// columns of dP and dP(t+1) waits until the writers have read it out.
// Every barrier is used once per block, so parities are (t & 1); no waiter can
// fall two phases behind because each producer waits on the consumer of its
// previous phase before it produces again.
//
// Every mbarrier wait is bounded; on expiry the CTA records the timeout in the
// status word, stops issuing, waits (bounded) for its loads and MMAs in flight,
// frees tensor memory and exits.
#include <algorithm>
#include <climits>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {

constexpr int kBwdEwWarps = 8;                    // warps 0-7: elementwise (warpgroups 0, 1)
constexpr int kBwdWarpDq0 = 8;                    // warps 8-11: dQ writers (warpgroup 2)
constexpr int kBwdWarpTma = 12, kBwdWarpMma = 13; // warpgroup 3 (warps 14, 15 idle)
constexpr int kBwdThreads = 16 * 32;
// Registers: the launch gives every thread 128 (65536 / 512).  Warpgroup 3 drops to
// 72 and the other three rise to 144; each SM sub-partition holds one warp of every
// warpgroup, and 3 x 144 + 72 = 504 <= 4 x 128 per thread slot.
constexpr uint32_t kBwdRegsLaunch = 128, kBwdRegsWork = 144, kBwdRegsIo = 72;
static_assert(3 * kBwdRegsWork + kBwdRegsIo <= 4 * kBwdRegsLaunch, "register split exceeds the launch");
static_assert(kBwdRegsLaunch * kBwdThreads <= 65536, "launch registers");

template <int D>
struct BwdCfg {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int kBlocks = D / 64;
    static constexpr int kBlockBytes = 128 * 128;      // one 64-column block of a 128-row tile
    static constexpr int kTileBytes = 128 * D * 2;     // a K, V, Q or dO tile
    static constexpr int kStages = 2;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kTileBytes;
    static constexpr int kOffQ = kOffV + kTileBytes;
    static constexpr int kOffDO = kOffQ + kStages * kTileBytes;
    static constexpr int kOffDS = kOffDO + kStages * kTileBytes;  // [128 keys][128 queries] 16-bit
    static constexpr int kDSBytes = 128 * 128 * 2;
    static constexpr int kOffVec = kOffDS + kDSBytes;             // per slot: lse2[128], D[128]
    static constexpr int kVecBytes = 2 * 128 * 4;
    static constexpr int kOffBar = kOffVec + kStages * kVecBytes;
    // barriers: kv, q_full[S], q_empty[S], do_full[S], do_empty[S], s_full, dp_full, p_ready,
    // ds_ready, dv_done, dq_full, dq_free, ds_free, final, mma_fin
    static constexpr int kNumBars = 1 + 4 * kStages + 10;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kBytes = kOffMisc + 16;
    // Slack to align the base to 1024 bytes when it fits; otherwise the kernel
    // requires (and checks) an aligned base.
    static constexpr int kSlack = (kBytes + 1024 <= 232448) ? 1024 : 0;
    static constexpr int kSmemBytes = kBytes + kSlack;
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
    static constexpr uint32_t kTmemS = 0, kTmemDP = 128, kTmemDV = 256, kTmemDK = 256 + D;
    static constexpr uint32_t kTmemDQ = (D == 128) ? 128u : 256u + 2u * D;
    static constexpr uint32_t kTmemCols = 512;
};

// P for one thread's key and 32 query columns: p = 2^(s scale log2(e) + nl2) with
// nl2 = -LSE log2(e) of each query row (-inf on rows that see no key).  MASKED adds
// the causal mask (query q sees key j when q >= qmin) and the ragged end of the keys.
template <bool MASKED>
__device__ __forceinline__ void bwd_p_chunk(const uint32_t (&sv)[32], const float *nl2, float sl2, int q_first,
                                            int qmin, bool key_ok, float *p) {
    const uint64_t sl2x2 = f2_make(sl2, sl2);
#pragma unroll
    for (int e4 = 0; e4 < 8; ++e4) {
        const float4 L = reinterpret_cast<const float4 *>(nl2)[e4];
        const float2 x01 = f2_split(ffma2(f2_make(__uint_as_float(sv[4 * e4]), __uint_as_float(sv[4 * e4 + 1])),
                                          sl2x2, f2_make(L.x, L.y)));
        const float2 x23 = f2_split(ffma2(f2_make(__uint_as_float(sv[4 * e4 + 2]), __uint_as_float(sv[4 * e4 + 3])),
                                          sl2x2, f2_make(L.z, L.w)));
        float v[4] = {ex2_approx(x01.x), ex2_approx(x01.y), ex2_approx(x23.x), ex2_approx(x23.y)};
        if constexpr (MASKED) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (!key_ok || q_first + 4 * e4 + u < qmin) v[u] = 0.f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) p[4 * e4 + u] = v[u];
    }
}

// VARLEN: a packed variable-length batch.  blockIdx.x indexes a work list of
// (sequence, key block) pairs (longest sequences first), blockIdx.y is the K/V head;
// q, o, dO are [total_q, H, d], k, v, dK, dV are [total_k, H_kv, d] (tensor maps
// indexed by column, head, token), and sequence s spans tokens [cu_q[s], cu_q[s+1])
// of q and [cu_k[s], cu_k[s+1]) of k and v.  A query block may run past its
// sequence into the next one's tokens: those rows' padded LSE entries are -inf, so
// they get P = 0 and add nothing; keys past the sequence are masked like a ragged
// K tail.  A CTA past the end of the work list leaves at entry.
template <int D, bool BF16, bool VARLEN>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                  const BwdArgs args) {
    using C = BwdCfg<D>;
    using PK = Pack<BF16>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    if (pad > (uint32_t)C::kSlack) {  // uniform over the CTA: nothing has been touched yet
        if (threadIdx.x == 0) atomicOr(args.status, kDevErrLayout);
        return;
    }
    uint8_t *smem = smem_raw + pad;
    const uint32_t sb = raw + pad;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int k0 = blockIdx.x * kBwdBc;  // first key of this block (block 0 has the most work when causal)
    const int causal = args.causal;
    const int H_kv = args.H / args.group;
    int Nq, Nk, bhk, bh0, ld_rows, seq_off, q_tok = 0, k_tok = 0;
    if constexpr (VARLEN) {
        if ((int)blockIdx.x >= args.work[0]) return;  // past the list: the whole CTA, nothing touched yet
        const int2 w = reinterpret_cast<const int2 *>(args.work + 2)[blockIdx.x];
        const int seq = w.x;
        k0 = w.y * kBwdBc;
        bhk = blockIdx.y;                      // K/V head within a token
        q_tok = args.cu_q[seq];
        k_tok = args.cu_k[seq];
        Nq = args.cu_q[seq + 1] - q_tok;
        Nk = args.cu_k[seq + 1] - k_tok;
        bh0 = bhk * args.group;                // first query head (within a token) of the group
        ld_rows = args.rows_pad;               // workspace rows per head
        seq_off = args.row_off[seq];           // this sequence's first workspace row
        if (k0 >= Nk) return;                  // the whole CTA: nothing has been touched yet
    } else {
        bhk = blockIdx.y;                      // K/V head (b * H_kv + h_kv)
        Nq = args.Nq;
        Nk = args.Nk;
        bh0 = (bhk / H_kv) * args.H + (bhk % H_kv) * args.group;  // first query head of the group
        ld_rows = args.Nq_pad;
        seq_off = 0;
    }
    // The query rows of head h (global for dense, within a token for VARLEN) and block
    // q0 sit at workspace rows h * ld_rows + seq_off + q0 ... (vectors and dQ accumulator).
    const int num_m = (Nq + kBwdBr - 1) / kBwdBr;
    // Query row q sees key k when k <= q + (Nk - Nq) under the causal mask, so the
    // first query block with a row that sees key k0 starts at row k0 - (Nk - Nq).
    int i_start = 0;
    if (causal) {
        const int first_q = k0 - (Nk - Nq);
        i_start = first_q <= 0 ? 0 : first_q / kBwdBr;
    }
    // Step t visits query block i_start + t % n_q of the (t / n_q)-th query head that
    // reads this K/V head (grouped-query attention: `group` consecutive query heads).
    const int n_q = max(0, num_m - i_start);
    const int n = n_q * args.group;
    // Each role walks the steps with a StepCursor: query block and query head of step t,
    // advanced by counting (no division in the loops).
    struct StepCursor {
        int q0, bh, ti, q0_first, n_q;
        __device__ __forceinline__ void next() {
            if (++ti == n_q) {
                ti = 0;
                q0 = q0_first;
                ++bh;
            } else {
                q0 += kBwdBr;
            }
        }
    };
    const StepCursor cursor0{i_start * kBwdBr, bh0, 0, i_start * kBwdBr, n_q};

    auto bar = [&](int idx) -> uint32_t { return sb + C::kOffBar + 8u * (uint32_t)idx; };
    constexpr int S_ = C::kStages;
    constexpr int B_KV = 0;
    auto B_QFULL = [](int s) { return 1 + s; };
    auto B_QEMPTY = [](int s) { return 1 + S_ + s; };
    auto B_DOFULL = [](int s) { return 1 + 2 * S_ + s; };
    auto B_DOEMPTY = [](int s) { return 1 + 3 * S_ + s; };
    constexpr int B_SFULL = 1 + 4 * S_;
    constexpr int B_DPFULL = B_SFULL + 1;
    constexpr int B_PREADY = B_SFULL + 2;   // one arrival per elementwise warp
    constexpr int B_DSREADY = B_SFULL + 3;  // one arrival per elementwise warp
    constexpr int B_DVDONE = B_SFULL + 4;
    constexpr int B_DQFULL = B_SFULL + 5;
    constexpr int B_DQFREE = B_SFULL + 6;   // one arrival per dQ-writer warp
    constexpr int B_DSFREE = B_SFULL + 7;
    constexpr int B_FINAL = B_SFULL + 8;
    constexpr int B_MMAFIN = B_SFULL + 9;
    volatile uint32_t *tmem_holder = reinterpret_cast<volatile uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
    int *status = args.status;

    if (threadIdx.x == 0) {
        mbar_init(bar(B_KV), 1);
        for (int s = 0; s < S_; ++s) {
            mbar_init(bar(B_QFULL(s)), 1);
            mbar_init(bar(B_QEMPTY(s)), 1);
            mbar_init(bar(B_DOFULL(s)), 1);
            mbar_init(bar(B_DOEMPTY(s)), 1);
        }
        mbar_init(bar(B_SFULL), 1);
        mbar_init(bar(B_DPFULL), 1);
        mbar_init(bar(B_PREADY), kBwdEwWarps);
        mbar_init(bar(B_DSREADY), kBwdEwWarps);
        mbar_init(bar(B_DVDONE), 1);
        mbar_init(bar(B_DQFULL), 1);
        mbar_init(bar(B_DQFREE), 4);
        mbar_init(bar(B_DSFREE), 1);
        mbar_init(bar(B_FINAL), 1);
        mbar_init(bar(B_MMAFIN), 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmDO);
    }
    if (warp == kBwdWarpMma) {
        tmem_alloc(sb + C::kOffMisc, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    constexpr uint32_t hi = sdesc_hi_sw128(1024);  // 8 rows x 128 B per core group

    if (warp >= kBwdWarpTma) {
      // Warpgroup 3: TMA producer and MMA issuer, one lane each.
      regs_decrease<kBwdRegsIo>();
      if (warp == kBwdWarpTma) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && n > 0) {
            uint32_t pend_q = 0, pend_do = 0, par_q = 0, par_do = 0;
            mbar_arrive_expect_tx(bar(B_KV), 2 * C::kTileBytes);
            for (int b = 0; b < C::kBlocks; ++b) {
                if constexpr (VARLEN) {
                    tma_load_3d(sb + C::kOffK + b * C::kBlockBytes, &tmK, b * 64, bhk, k_tok + k0, bar(B_KV));
                    tma_load_3d(sb + C::kOffV + b * C::kBlockBytes, &tmV, b * 64, bhk, k_tok + k0, bar(B_KV));
                } else {
                    tma_load_3d(sb + C::kOffK + b * C::kBlockBytes, &tmK, b * 64, k0, bhk, bar(B_KV));
                    tma_load_3d(sb + C::kOffV + b * C::kBlockBytes, &tmV, b * 64, k0, bhk, bar(B_KV));
                }
            }
            bool ok = true;
            StepCursor cur = cursor0;
            for (int t = 0; ok && t < n; ++t, cur.next()) {
                const int s = t % S_;
                const uint32_t it = (uint32_t)(t / S_);
                const int q0 = cur.q0, bh = cur.bh;
                const size_t vec_row = (size_t)bh * ld_rows + seq_off;
                // Q and dO rows: (row, head) for dense tensors, (head, token) for packed ones
                const int qy = VARLEN ? bh : q0, qz = VARLEN ? q_tok + q0 : bh;
                ok = mbar_wait_bounded(bar(B_QEMPTY(s)), (it & 1u) ^ 1u, abort_flag, status);
                if (!ok) break;
                mbar_arrive_expect_tx(bar(B_QFULL(s)), C::kTileBytes + C::kVecBytes);
                for (int b = 0; b < C::kBlocks; ++b)
                    tma_load_3d(sb + C::kOffQ + s * C::kTileBytes + b * C::kBlockBytes, &tmQ, b * 64, qy, qz,
                                bar(B_QFULL(s)));
                const uint32_t vdst = sb + C::kOffVec + s * C::kVecBytes;
                bulk_load(vdst, args.lse2 + vec_row + q0, 512, bar(B_QFULL(s)));
                bulk_load(vdst + 512, args.dvec + vec_row + q0, 512, bar(B_QFULL(s)));
                pend_q |= 1u << s;
                par_q = (par_q & ~(1u << s)) | ((it & 1u) << s);
                ok = mbar_wait_bounded(bar(B_DOEMPTY(s)), (it & 1u) ^ 1u, abort_flag, status);
                if (!ok) break;
                mbar_arrive_expect_tx(bar(B_DOFULL(s)), C::kTileBytes);
                for (int b = 0; b < C::kBlocks; ++b)
                    tma_load_3d(sb + C::kOffDO + s * C::kTileBytes + b * C::kBlockBytes, &tmDO, b * 64, qy, qz,
                                bar(B_DOFULL(s)));
                pend_do |= 1u << s;
                par_do = (par_do & ~(1u << s)) | ((it & 1u) << s);
            }
            // Every load issued must land before the CTA may exit.
            volatile int no_abort = 0;
            mbar_wait_bounded(bar(B_KV), 0, &no_abort, status);
            for (int s = 0; s < S_; ++s) {
                if (pend_q & (1u << s)) mbar_wait_bounded(bar(B_QFULL(s)), (par_q >> s) & 1u, &no_abort, status);
                if (pend_do & (1u << s)) mbar_wait_bounded(bar(B_DOFULL(s)), (par_do >> s) & 1u, &no_abort, status);
            }
        }
      } else if (warp == kBwdWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n > 0) {
            constexpr uint32_t idesc_s = idesc_f16(128, 128, BF16, false, false);  // S^T, dP^T
            constexpr uint32_t idesc_kv = idesc_f16(128, D, BF16, true, false);    // dV, dK
            constexpr uint32_t idesc_q = (D == 128) ? idesc_f16(128, 128, BF16, true, true)  // dQ^T
                                                    : idesc_f16(128, 64, BF16, true, true);  // dQ
            const uint32_t k_lo = sdesc_lo(sb + C::kOffK, 16);                  // K-major: LBO unused
            const uint32_t v_lo = sdesc_lo(sb + C::kOffV, 16);
            const uint32_t k_mn = sdesc_lo(sb + C::kOffK, C::kBlockBytes);      // MN-major: LBO = block
            const uint32_t ds_k = sdesc_lo(sb + C::kOffDS, 16);
            const uint32_t ds_mn = sdesc_lo(sb + C::kOffDS, C::kBlockBytes);
            // S^T(t) = K Q_t^T into [0,128).
            auto issue_s = [&](int t) {
                const uint32_t q_lo = sdesc_lo(sb + C::kOffQ + (t % S_) * C::kTileBytes, 16);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (uint32_t)((k >> 2) * C::kBlockBytes + (k & 3) * 32) >> 4;
                    umma_ss_w(tmem + C::kTmemS, k_lo + off, hi, q_lo + off, hi, idesc_s, k > 0 ? 1u : 0u);
                }
                umma_commit(bar(B_SFULL));
            };
            bool ok = mbar_wait_bounded(bar(B_KV), 0, abort_flag, status) &&
                      mbar_wait_bounded(bar(B_QFULL(0)), 0, abort_flag, status);
            if (ok) {
                tc_fence_after();
                issue_s(0);
            }
            for (int t = 0; ok && t < n; ++t) {
                const int s = t % S_;
                const uint32_t ph = (uint32_t)(t / S_) & 1u;
                const uint32_t pt = (uint32_t)t & 1u, pp = (uint32_t)(t - 1) & 1u;
                // dP^T(t) = V dO_t^T into [128,256); for d = 128 once dQ^T(t-1) has been read out.
                ok = mbar_wait_bounded(bar(B_DOFULL(s)), ph, abort_flag, status) &&
                     (D != 128 || t == 0 || mbar_wait_bounded(bar(B_DQFREE), pp, abort_flag, status));
                if (!ok) break;
                tc_fence_after();
                const uint32_t do_lo = sdesc_lo(sb + C::kOffDO + s * C::kTileBytes, 16);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (uint32_t)((k >> 2) * C::kBlockBytes + (k & 3) * 32) >> 4;
                    umma_ss_w(tmem + C::kTmemDP, v_lo + off, hi, do_lo + off, hi, idesc_s, k > 0 ? 1u : 0u);
                }
                umma_commit(bar(B_DPFULL));
                // dV += P^T dO_t: P^T from tensor memory, 16 queries per instruction.
                ok = mbar_wait_bounded(bar(B_PREADY), pt, abort_flag, status);
                if (!ok) break;
                tc_fence_after();
                const uint32_t do_mn = sdesc_lo(sb + C::kOffDO + s * C::kTileBytes, C::kBlockBytes);
#pragma unroll
                for (int k = 0; k < kBwdBr / 16; ++k)
                    umma_ts_w(tmem + C::kTmemDV, tmem + C::kTmemS + 64 * (k >> 2) + 8 * (k & 3),
                              do_mn + (uint32_t)((k * 2048) >> 4), hi, idesc_kv, (t > 0 || k > 0) ? 1u : 0u);
                umma_commit(bar(B_DVDONE));
                umma_commit(bar(B_DOEMPTY(s)));
                // S^T(t+1) next, so that the elementwise warps can start on P(t+1) while the
                // tensor core does dK(t) and dQ(t); it overwrites P(t) once dV(t) completed.
                if (t + 1 < n) {
                    ok = mbar_wait_bounded(bar(B_QFULL((t + 1) % S_)), (uint32_t)((t + 1) / S_) & 1u, abort_flag,
                                           status) &&
                         mbar_wait_bounded(bar(B_DVDONE), pt, abort_flag, status);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(t + 1);
                }
                // dK += dS^T Q_t.
                ok = mbar_wait_bounded(bar(B_DSREADY), pt, abort_flag, status);
                if (!ok) break;
                tc_fence_after();
                const uint32_t q_mn = sdesc_lo(sb + C::kOffQ + s * C::kTileBytes, C::kBlockBytes);
#pragma unroll
                for (int k = 0; k < kBwdBr / 16; ++k) {
                    const uint32_t off = (uint32_t)((k >> 2) * C::kBlockBytes + (k & 3) * 32) >> 4;
                    umma_ss_w(tmem + C::kTmemDK, ds_k + off, hi, q_mn + (uint32_t)((k * 2048) >> 4), hi, idesc_kv,
                              (t > 0 || k > 0) ? 1u : 0u);
                }
                umma_commit(bar(B_QEMPTY(s)));
                // dQ(t): for d = 64 into its own columns, once dQ(t-1) has been read out.
                if (D != 128 && t > 0) {
                    ok = mbar_wait_bounded(bar(B_DQFREE), pp, abort_flag, status);
                    if (!ok) break;
                    tc_fence_after();
                }
#pragma unroll
                for (int k = 0; k < kBwdBc / 16; ++k) {
                    const uint32_t off = (uint32_t)((k * 2048) >> 4);  // 16 keys of 128-byte rows
                    if constexpr (D == 128)
                        umma_ss_w(tmem + C::kTmemDQ, k_mn + off, hi, ds_mn + off, hi, idesc_q, k > 0 ? 1u : 0u);
                    else
                        umma_ss_w(tmem + C::kTmemDQ, ds_mn + off, hi, k_mn + off, hi, idesc_q, k > 0 ? 1u : 0u);
                }
                umma_commit(bar(B_DQFULL));
                umma_commit(bar(B_DSFREE));
            }
            if (ok) umma_commit(bar(B_FINAL));
            // Tensor memory may be freed only after every issued MMA completed.
            umma_commit(bar(B_MMAFIN));
            volatile int no_abort = 0;
            mbar_wait_bounded(bar(B_MMAFIN), 0, &no_abort, status);
        }
      }
    } else if (warp >= kBwdWarpDq0) {
        // ------------------------------------------------------------ dQ writers
        // All of dQ(t) is read from tensor memory at once (its columns are released for
        // dP(t+1) right away), then summed into the fp32 accumulator.
        regs_increase<kBwdRegsWork>();
        const int qw = warp & 3;
        const uint32_t lane_base = tmem + ((uint32_t)(qw * 32) << 16);
        bool ok = true;
        StepCursor cur = cursor0;
        for (int t = 0; t < n; ++t, cur.next()) {
            const int q0 = cur.q0, bh = cur.bh;
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(B_DQFULL), (uint32_t)t & 1u, abort_flag, status));
            if (!ok) break;
            tc_fence_after();
            if constexpr (D == 128) {
                // dQ^T: lane = head-dim index, columns = the block's 128 queries; a warp's
                // 32 lanes add to 32 consecutive floats of one dQ row.
                uint32_t a[128];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t (&ac)[32] = *reinterpret_cast<uint32_t(*)[32]>(a + 32 * c);
                    tmem_ld_32x32b_x32(lane_base + C::kTmemDQ + 32 * c, ac);
                }
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_DQFREE));
                float *dst = args.dq_acc + ((size_t)bh * ld_rows + seq_off + q0) * 128 + qw * 32 + lane;
                const int rows = Nq - q0;
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c < rows) atomicAdd(dst + (size_t)c * 128, __uint_as_float(a[c]));
            } else {
                // dQ: lane = query row q0 + 32 qw + lane, columns = the 64 head-dim indices.
                uint32_t a[64];
                tmem_ld_32x32b_x32(lane_base + C::kTmemDQ, *reinterpret_cast<uint32_t(*)[32]>(a));
                tmem_ld_32x32b_x32(lane_base + C::kTmemDQ + 32, *reinterpret_cast<uint32_t(*)[32]>(a + 32));
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_DQFREE));
                const int q = q0 + qw * 32 + lane;
                if (q < Nq) {
                    float4 *dst = reinterpret_cast<float4 *>(args.dq_acc + ((size_t)bh * ld_rows + seq_off + q) * 64);
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        atomicAdd(dst + e, make_float4(__uint_as_float(a[4 * e]), __uint_as_float(a[4 * e + 1]),
                                                       __uint_as_float(a[4 * e + 2]), __uint_as_float(a[4 * e + 3])));
                }
            }
        }
    } else {
        // ------------------------------------------------------------ elementwise and epilogue
        regs_increase<kBwdRegsWork>();
        const int qw = warp & 3;  // TMEM lanes [32 qw, 32 qw + 32)
        const int g = warp >> 2;  // query columns [64 g, 64 g + 64) of each block
        const int r = qw * 32 + lane;
        const int j = k0 + r;     // this thread's key
        const bool key_ok = j < Nk;
        const int qmin = causal ? j - (Nk - Nq) : INT_MIN;  // the first query row that sees key j
        const bool tail_block = k0 + kBwdBc > Nk;
        const uint32_t lane_base = tmem + ((uint32_t)(qw * 32) << 16);
        const float sl2 = args.scale_log2;
        float p[64];
        bool ok = true;
        StepCursor cur = cursor0;
        for (int t = 0; t < n; ++t, cur.next()) {
            const int s = t % S_;
            const uint32_t pt = (uint32_t)t & 1u;
            const int q0 = cur.q0;
            const bool masked = tail_block || (causal && (q0 + (Nk - Nq) < k0 + kBwdBc - 1));
            // ---- P = 2^(S scale log2(e) - LSE log2(e)) for this thread's key and 64 queries
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(B_QFULL(s)), (uint32_t)(t / S_) & 1u, abort_flag,
                                                           status) &&
                                             mbar_wait_bounded(bar(B_SFULL), pt, abort_flag, status));
            if (!ok) break;
            tc_fence_after();
            const float *nl2 = reinterpret_cast<const float *>(smem + C::kOffVec + s * C::kVecBytes);
            const float *ndv = nl2 + 128;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t sv[32];
                tmem_ld_32x32b_x32(lane_base + C::kTmemS + 64 * g + 32 * cc, sv);
                tmem_wait_ld();
                const int col = 64 * g + 32 * cc;
                if (masked)
                    bwd_p_chunk<true>(sv, nl2 + col, sl2, q0 + col, qmin, key_ok, p + 32 * cc);
                else
                    bwd_p_chunk<false>(sv, nl2 + col, sl2, q0 + col, qmin, key_ok, p + 32 * cc);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) pk[e] = PK::pack(p[32 * cc + 2 * e], p[32 * cc + 2 * e + 1]);
                // These columns' scores were read above: the 16-bit pairs go over them.
                tmem_st_32x32b_x16(lane_base + C::kTmemS + 64 * g + 16 * cc, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_PREADY));
            // ---- dS = P (dP - D), to shared memory [key][query] (128-byte swizzle)
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(B_DPFULL), pt, abort_flag, status) &&
                                             (t == 0 || mbar_wait_bounded(bar(B_DSFREE), pt ^ 1u, abort_flag, status)));
            if (!ok) break;
            tc_fence_after();
            uint8_t *ds_row = smem + C::kOffDS + g * C::kBlockBytes + r * 128;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t dp[32];
                tmem_ld_32x32b_x32(lane_base + C::kTmemDP + 64 * g + 32 * cc, dp);
                tmem_wait_ld();
                const float4 *d4 = reinterpret_cast<const float4 *>(ndv + 64 * g + 32 * cc);
                uint32_t pk[16];
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4) {
                    const float4 Dv = d4[e4];
                    const int c = 32 * cc + 4 * e4;
                    const float2 d01 = f2_split(fmul2(f2_make(p[c], p[c + 1]),
                                                      fadd2(f2_make(__uint_as_float(dp[4 * e4]), __uint_as_float(dp[4 * e4 + 1])),
                                                            f2_make(Dv.x, Dv.y))));
                    const float2 d23 = f2_split(fmul2(f2_make(p[c + 2], p[c + 3]),
                                                      fadd2(f2_make(__uint_as_float(dp[4 * e4 + 2]), __uint_as_float(dp[4 * e4 + 3])),
                                                            f2_make(Dv.z, Dv.w))));
                    pk[2 * e4] = PK::pack(d01.x, d01.y);
                    pk[2 * e4 + 1] = PK::pack(d23.x, d23.y);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int chunk = 4 * cc + u;  // 8 queries of 16 bits each
                    *reinterpret_cast<uint4 *>(ds_row + ((chunk ^ (r & 7)) << 4)) =
                        make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_DSREADY));
        }
        if (ok && n > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(B_FINAL), 0, abort_flag, status));
            tc_fence_after();
        }
        if (ok) {
            // Epilogue: this warp's half of the head dimension of dV_j and dK_j = scale * acc.
            // The tensor-memory loads are warp-collective: every lane takes part, and
            // only lanes whose key exists store.
            const size_t orow = VARLEN ? ((size_t)(k_tok + j) * H_kv + bhk) * D : ((size_t)bhk * Nk + j) * D;
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
                typename PK::T *dst_row = reinterpret_cast<typename PK::T *>(which == 0 ? args.dv : args.dk) + orow;
                const uint32_t src = lane_base + (which == 0 ? C::kTmemDV : C::kTmemDK);
                const float f = which == 0 ? 1.f : args.scale;
#pragma unroll 1
                for (int c = 0; c < D / 64; ++c) {
                    const int col = g * (D / 2) + 32 * c;
                    uint32_t v[32];
                    if (n > 0) {
                        tmem_ld_32x32b_x32(src + col, v);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = 0u;
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = PK::pack(__uint_as_float(v[2 * e]) * f, __uint_as_float(v[2 * e + 1]) * f);
                    if (key_ok) {
                        uint4 *dst = reinterpret_cast<uint4 *>(dst_row + col);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kBwdWarpMma) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// Largest s in [0, n] with a[s] <= x, for a non-decreasing a with a[0] <= x: the
// sequence that holds token (or workspace row) x, skipping empty sequences.
__device__ __forceinline__ int seq_of(const int *a, int n, int x) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Variable-length batches: row_off[s] = sum over s' < s of ceil(len_q(s') / 128) * 128,
// the first workspace row of sequence s (s = 0 .. num_seqs).  One warp.
__global__ void fa_bwd_plan_kernel(const BwdArgs a) {
    const int lane = threadIdx.x;
    int base = 0;
    if (lane == 0) a.row_off[0] = 0;
    for (int s0 = 0; s0 < a.num_seqs; s0 += 32) {
        const int s = s0 + lane;
        int v = s < a.num_seqs ? (a.cu_q[s + 1] - a.cu_q[s] + kBwdBr - 1) / kBwdBr * kBwdBr : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
        if (s < a.num_seqs) a.row_off[s + 1] = base + v;
        base += __shfl_sync(0xffffffffu, v, 31);
    }
}

// -D_i = -dO_i . O_i (fp32), -lse2_i = -LSE_i log2(e) (-inf where LSE_i = -inf and
// on the padding rows, so that P = 2^(x - lse2) = 0 there), and the row of the dQ
// accumulator zeroed.  One warp per workspace row: [BH][Nq_pad] (dense; rows
// q >= Nq are padding) or [H][rows_pad] (VARLEN; row row_off[s] + r holds token
// cu_q[s] + r when r < len_q(s), every other row is padding).
template <int D, bool BF16, bool VARLEN>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const BwdArgs a) {
    using PK = Pack<BF16>;
    const int lane = threadIdx.x & 31;
    const int ld = VARLEN ? a.rows_pad : a.Nq_pad;
    const long long rows = (long long)a.BH * ld;
    const long long stride = (long long)gridDim.x * 8;
    for (long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); row < rows; row += stride) {
        const int bh = (int)(row / ld), q = (int)(row % ld);
        float4 *acc = reinterpret_cast<float4 *>(a.dq_acc + row * D);
        if (lane < D / 4) acc[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
        bool real;
        size_t off, lse_idx;
        if constexpr (VARLEN) {
            const int s = seq_of(a.row_off, a.num_seqs, q);
            const int r = q - a.row_off[s];
            real = s < a.num_seqs && r < a.cu_q[s + 1] - a.cu_q[s];
            const int tok = real ? a.cu_q[s] + r : 0;
            off = ((size_t)tok * a.BH + bh) * D;         // [total_q, H, d]
            lse_idx = (size_t)bh * a.total_q + tok;     // [H, total_q]
        } else {
            real = q < a.Nq;
            off = ((size_t)bh * a.Nq + q) * D;
            lse_idx = (size_t)bh * a.Nq + q;
        }
        float dot = 0.f, l2 = INFINITY;
        if (real) {
            const uint32_t *o32 = reinterpret_cast<const uint32_t *>(static_cast<const typename PK::T *>(a.o) + off);
            const uint32_t *g32 = reinterpret_cast<const uint32_t *>(static_cast<const typename PK::T *>(a.dout) + off);
#pragma unroll
            for (int e = 0; e < D / 64; ++e) {
                const float2 ov = PK::unpack(o32[lane + 32 * e]);
                const float2 gv = PK::unpack(g32[lane + 32 * e]);
                dot = fmaf(ov.x, gv.x, fmaf(ov.y, gv.y, dot));
            }
#pragma unroll
            for (int sft = 16; sft > 0; sft >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, sft);
            const float lse = a.lse[lse_idx];
            l2 = (lse == -INFINITY) ? INFINITY : lse * 1.4426950408889634f;
        }
        if (lane == 0) {  // stored negated: the main kernel adds them
            a.dvec[row] = -dot;
            a.lse2[row] = -l2;
        }
    }
}

// dQ = scale * accumulator, rounded to 16 bits; four elements per thread step.
// Output rows: [BH][Nq] (dense) or [total_q][H] (VARLEN).
template <int D, bool BF16, bool VARLEN>
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const BwdArgs a) {
    using PK = Pack<BF16>;
    const long long nrows = VARLEN ? (long long)a.total_q * a.BH : (long long)a.BH * a.Nq;
    const long long n4 = nrows * (D / 4);
    for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < n4; x += (long long)gridDim.x * blockDim.x) {
        const long long row = x / (D / 4);
        const int c4 = (int)(x % (D / 4));
        size_t acc_row;
        if constexpr (VARLEN) {
            const int tok = (int)(row / a.BH), h = (int)(row % a.BH);
            const int s = seq_of(a.cu_q, a.num_seqs, tok);
            acc_row = (size_t)h * a.rows_pad + a.row_off[s] + (tok - a.cu_q[s]);
        } else {
            const int bh = (int)(row / a.Nq), q = (int)(row % a.Nq);
            acc_row = (size_t)bh * a.Nq_pad + q;
        }
        const float4 v = reinterpret_cast<const float4 *>(a.dq_acc + acc_row * D)[c4];
        uint2 out;
        out.x = PK::pack(v.x * a.scale, v.y * a.scale);
        out.y = PK::pack(v.z * a.scale, v.w * a.scale);
        reinterpret_cast<uint2 *>(static_cast<typename PK::T *>(a.dq) + (size_t)row * D)[c4] = out;
    }
}

template <int D, bool BF16, bool VARLEN>
static cudaError_t launch_bwd_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                                const CUtensorMap &tdo, const BwdArgs &a_in, int *work, int capacity,
                                cudaStream_t stream) {
    BwdArgs a = a_in;
    a.work = work;
    using C = BwdCfg<D>;
    cudaError_t e;
    if constexpr (VARLEN) {
        e = launch_kernel(fa_bwd_plan_kernel, dim3(1), dim3(32), 0, stream, a);
        if (e != cudaSuccess) return e;
        e = launch_varlen_plan(a.cu_k, a.num_seqs, work, false, stream);
        if (e != cudaSuccess) return e;
    }
    const long long rows = (long long)a.BH * (VARLEN ? a.rows_pad : a.Nq_pad);
    const unsigned prep_blocks = (unsigned)std::min<long long>((rows + 7) / 8, 152LL * 64);
    e = launch_kernel(fa_bwd_prep_kernel<D, BF16, VARLEN>, dim3(prep_blocks), dim3(256), 0, stream, a);
    if (e != cudaSuccess) return e;
    auto kern = fa_bwd_kernel<D, BF16, VARLEN>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int H_kv = a.H / a.group;
    const dim3 grid = VARLEN ? dim3((unsigned)capacity, (unsigned)H_kv, 1)
                             : dim3((unsigned)((a.Nk + kBwdBc - 1) / kBwdBc), (unsigned)(a.BH / a.group), 1);
    e = launch_kernel(kern, grid, dim3(kBwdThreads), C::kSmemBytes, stream, tq, tk, tv, tdo, a);
    if (e != cudaSuccess) return e;
    const long long n4 = (VARLEN ? (long long)a.total_q * a.BH : (long long)a.BH * a.Nq) * (D / 4);
    const unsigned dq_blocks = (unsigned)std::min<long long>(std::max<long long>((n4 + 255) / 256, 1), 152LL * 64);
    return launch_kernel(fa_bwd_dq_kernel<D, BF16, VARLEN>, dim3(dq_blocks), dim3(256), 0, stream, a);
}

cudaError_t launch_bwd(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &tdo, const BwdArgs &a, cudaStream_t stream) {
    if (d == 64) return bf16 ? launch_bwd_t<64, true, false>(tq, tk, tv, tdo, a, nullptr, 0, stream)
                             : launch_bwd_t<64, false, false>(tq, tk, tv, tdo, a, nullptr, 0, stream);
    return bf16 ? launch_bwd_t<128, true, false>(tq, tk, tv, tdo, a, nullptr, 0, stream)
                : launch_bwd_t<128, false, false>(tq, tk, tv, tdo, a, nullptr, 0, stream);
}

cudaError_t launch_bwd_varlen(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                              const CUtensorMap &tdo, const BwdArgs &a, int *work, int capacity, cudaStream_t stream) {
    if (d == 64) return bf16 ? launch_bwd_t<64, true, true>(tq, tk, tv, tdo, a, work, capacity, stream)
                             : launch_bwd_t<64, false, true>(tq, tk, tv, tdo, a, work, capacity, stream);
    return bf16 ? launch_bwd_t<128, true, true>(tq, tk, tv, tdo, a, work, capacity, stream)
                : launch_bwd_t<128, false, true>(tq, tk, tv, tdo, a, work, capacity, stream);
}

}  // namespace fa
