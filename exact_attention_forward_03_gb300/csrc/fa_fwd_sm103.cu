// fa_fwd_sm103.cu -- fused exact attention forward on sm_103a tensor cores.
//
// One CTA computes two 128-row Q tiles (A and B, 256 consecutive query rows) of
// one (batch, head):
//   O_i = sum_j softmax_j(scale * q_i . k_j + mask) v_j,  LSE_i = m_i + ln l_i
// following the FlashAttention-2 forward ("6.2 FlashAttention V2 explained",
// §6): the Q tiles stay on chip, K/V tiles stream past them, a running row max
// m and row sum l are kept per row, the accumulator is rescaled by
// exp(m_old - m_new) and divided by l once at the end (§3.2; "02 · FA2", §1).
// Causal masking visits only K/V tiles up to the diagonal and masks
// element-wise only on tiles that straddle it or the ragged Nk tail (§5.3;
// "02 · FA2", §4).
//
// Roles (warp specialisation, 10 warps):
//   warps 0-3  softmax of Q tile A, one thread per query row (TMEM lane = row)
//   warps 4-7  softmax of Q tile B
//   warp 8     TMA producer: both Q tiles and K_0 once, then one ring stage per
//              step j holding V_j and K_{j+1} (64 keys each)
//   warp 9     owns tensor memory; one lane issues every tcgen05.mma
//
// Tensor memory (512 columns), for each tile X: S_X (64 fp32 columns), two P
// buffers P_X[0], P_X[1] (64 keys as 16-bit pairs, 32 columns each) and O_X (d
// fp32 columns).  Because P has its own columns, S_X(j+1) = Q_X K_{j+1}^T is
// issued as soon as the softmax warps have read S_X(j) into registers, before
// O_X += P_X(j) V_j: the tensor core computes the next scores while the
// softmax of the current step runs, and the two tiles keep it fed.  Step j
// writes P_X[j % 2], so the softmax of step j waits only for the MMA that read
// that buffer two steps earlier.  MMA order per step j: S_A(j+1), S_B(j+1),
// PV_A(j), PV_B(j).
//
// On steps that need a mask, P is written as a 16-bit head P plus a 16-bit
// remainder P - P_head in the other buffer, and both are multiplied into O:
// rows near the diagonal see few keys, so one 16-bit rounding of their few
// large weights would otherwise dominate their error.  Every MMA group that
// reads a P buffer commits to that buffer's barrier, and both sides count those
// uses the same way, so the softmax always knows which phase to wait for.
//
// The two tiles share the barriers of the per-step handshakes (S ready, S read,
// P ready): the MMA warp waits once per step for both tiles, which keeps its
// serial bookkeeping between MMA groups short.  A tile with fewer steps than
// its partner keeps arriving on those barriers, paced by "S ready", until the
// partner is done.
//
// The rescale of O by alpha = 2^(m_old - m_new) is done only when the row max
// of some row in the warp grew by more than 2^8: otherwise m stays and p may
// reach 2^8, which changes nothing in exact arithmetic (O and l share the same
// stale max) and keeps fp16/bf16/fp32 far from overflow.
//
// Every mbarrier wait is bounded (%globaltimer); on expiry the CTA records
// the timeout in the status word, stops issuing work, waits (bounded) for its
// in-flight TMA loads and MMAs, frees tensor memory and exits.
#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {

constexpr int kFwdThreads = 320;
constexpr int kWarpTma = 8, kWarpMma = 9;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct FwdCfg {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int kBlocks = D / 64;               // 128-byte swizzle blocks per row
    static constexpr int kQBlockBytes = kFwdBr * 128;    // one 64-column block of a Q tile
    static constexpr int kKVBlockBytes = kFwdBc * 128;   // one 64-column block of a K/V tile
    static constexpr int kQBytes = kFwdBr * D * 2;       // one Q tile
    static constexpr int kTileBytes = kFwdBc * D * 2;    // one K or V tile
    static constexpr int kStages = (D == 128) ? 4 : 8;  // ring stages of (V_j, K_{j+1})
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kOffQ = 0;                      // Q_A, then Q_B
    static constexpr int kOffK0 = kFwdTilesPerCta * kQBytes;
    static constexpr int kOffRing = kOffK0 + kTileBytes;
    static constexpr int kOffBar = kOffRing + kStages * kStageBytes;
    // barriers: q_full, full[S], empty[S], s_full, s_free, p_full[2], p_read[2][2], o_final[2], mma_fin
    static constexpr int kNumBars = 1 + 2 * kStages + 1 + 1 + 2 + 4 + 2 + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack to align the base to 1024
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
    static constexpr uint32_t kTmemCols = 512;
    __device__ static constexpr uint32_t tmem_s(int x) { return 64u * x; }          // [0,64), [64,128)
    __device__ static constexpr uint32_t tmem_p(int x, int b) { return 128u + 64u * x + 32u * b; }  // [128,256)
    __device__ static constexpr uint32_t tmem_o(int x) { return 256u + (uint32_t)D * x; }
};

// Step j needs element masks when it crosses the ragged end of K or, under
// causal masking, holds a key beyond the first row's last visible key.
__device__ __forceinline__ bool fwd_tile_needs_mask(int j, int q0, int Nq, int Nk, int causal) {
    const int last_key = (j + 1) * kFwdBc - 1;
    return (last_key >= Nk) || (causal && last_key > q0 + (Nk - Nq));
}

// K/V steps that Q rows [q0, q0+128) must visit (0 when the tile holds no row).
__device__ __forceinline__ int fwd_tile_count(int q0, int Nq, int Nk, int causal) {
    if (q0 >= Nq) return 0;
    int kv_end = Nk;
    if (causal) kv_end = min(Nk, min(q0 + kFwdBr, Nq) + (Nk - Nq));
    return kv_end > 0 ? (kv_end + kFwdBc - 1) / kFwdBc : 0;
}

// O_X (32 rows of this warp, kCols columns) *= alpha, 16 columns at a time.
// Rarely taken (only when a row max grows by more than 2^8), so it is kept out
// of line to leave the registers of the common path alone.
template <int kCols>
__device__ __noinline__ void rescale_o(uint32_t o_addr, float alpha) {
    const uint64_t a2 = f2_make(alpha, alpha);
#pragma unroll 1
    for (int c = 0; c < kCols / 16; ++c) {
        uint32_t orow[16];
        tmem_ld_32x32b_x16(o_addr + 16 * c, orow);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
            const float2 v = f2_split(fmul2(f2_make(__uint_as_float(orow[e]), __uint_as_float(orow[e + 1])), a2));
            orow[e] = __float_as_uint(v.x);
            orow[e + 1] = __float_as_uint(v.y);
        }
        tmem_st_32x32b_x16(o_addr + 16 * c, orow);
    }
}

// One online-softmax step for the 64 S values of this thread's row held in
// `sr` (fp32 bits): optional causal/tail mask, (conditional) max update,
// p = 2^(s*c - m), the row sum, and P packed into 16-bit pairs in `ph` (plus
// the 16-bit remainder in `pl` on masked tiles).  Returns whether the warp
// moved its max; `alpha` is then the factor O and l are scaled by.
template <bool MASKED, bool BF16>
__device__ __forceinline__ bool softmax_step(uint32_t (&sr)[64], int c0, int lim, float sl2, float &m, float &l,
                                             float &alpha, uint32_t (&ph)[32], uint32_t (&pl)[32]) {
    using PK = Pack<BF16>;
    if (MASKED) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
            if (c0 + c > lim) sr[c] = __float_as_uint(-INFINITY);
    }
    float mx[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) mx[e] = fmax3(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1]), -INFINITY);
#pragma unroll
    for (int c = 16; c < 64; c += 2)
        mx[(c >> 1) & 7] = fmax3(mx[(c >> 1) & 7], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
    const float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
    const float m_cand = fmaxf(m, mt * sl2);
    const bool rescale = __any_sync(0xffffffffu, m_cand > m + kRescaleThreshold);
    alpha = 1.f;
    if (rescale) {
        const float m_new_d = (m_cand == -INFINITY) ? 0.f : m_cand;  // never subtract -inf from -inf
        alpha = ex2_approx(m - m_new_d);
        m = m_cand;
    }
    const float m_d = (m == -INFINITY) ? 0.f : m;
    const uint64_t scale2 = f2_make(sl2, sl2);
    const uint64_t shift2 = f2_make(-m_d, -m_d);
    uint64_t rs2[2] = {f2_make(0.f, 0.f), f2_make(0.f, 0.f)};
#pragma unroll
    for (int e = 0; e < 64; e += 2) {
        const float2 xa = f2_split(ffma2(f2_make(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), scale2, shift2));
        const float p0 = ex2_approx(xa.x);
        const float p1 = ex2_approx(xa.y);
        rs2[(e >> 1) & 1] = fadd2(rs2[(e >> 1) & 1], f2_make(p0, p1));
        ph[e >> 1] = PK::pack(p0, p1);
        if (MASKED) {
            const float2 hf = PK::unpack(ph[e >> 1]);
            pl[e >> 1] = PK::pack(p0 - hf.x, p1 - hf.y);
        }
    }
    const float2 r0 = f2_split(rs2[0]), r1 = f2_split(rs2[1]);
    l = l * alpha + ((r0.x + r0.y) + (r1.x + r1.y));
    return rescale;
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdArgs args) {
    using C = FwdCfg<D>;
    using PK = Pack<BF16>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sb = raw + pad;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Consecutive CTAs take consecutive row blocks of one head, heaviest causal
    // block first, so the CTAs resident at any time share a few heads' K/V in L2.
    const int bh = blockIdx.y;
    const int q0 = (args.num_m - 1 - (int)blockIdx.x) * (kFwdTilesPerCta * kFwdBr);
    const int Nq = args.Nq, Nk = args.Nk, causal = args.causal;
    const int nA = fwd_tile_count(q0, Nq, Nk, causal);
    const int nB = fwd_tile_count(q0 + kFwdBr, Nq, Nk, causal);
    const int n_max = max(nA, nB);

    auto bar = [&](int idx) -> uint32_t { return sb + C::kOffBar + 8u * (uint32_t)idx; };
    constexpr int B_QFULL = 0;
    auto B_FULL = [](int s) { return 1 + s; };
    auto B_EMPTY = [](int s) { return 1 + C::kStages + s; };
    constexpr int B_SFULL = 1 + 2 * C::kStages;  // S_A(j), S_B(j) ready
    constexpr int B_SFREE = 2 + 2 * C::kStages;  // both tiles have read S(j)
    // P[b] written by both tiles: one barrier per buffer, so the softmax (which may
    // run a step ahead of the MMA warp) can never complete a phase twice unseen.
    auto B_PFULL = [](int b) { return 3 + 2 * C::kStages + b; };
    auto B_PREAD = [](int x, int b) { return 5 + 2 * C::kStages + 2 * x + b; };  // an MMA group read P_X[b]
    auto B_OFINAL = [](int x) { return 9 + 2 * C::kStages + x; };
    constexpr int B_MMAFIN = 11 + 2 * C::kStages;
    volatile uint32_t *tmem_holder = reinterpret_cast<volatile uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
    int *status = args.status;

    if (threadIdx.x == 0) {
        mbar_init(bar(B_QFULL), 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar(B_FULL(s)), 1);
            mbar_init(bar(B_EMPTY(s)), 1);
        }
        mbar_init(bar(B_SFULL), 1);
        mbar_init(bar(B_SFREE), 256);
        mbar_init(bar(B_PFULL(0)), 256);
        mbar_init(bar(B_PFULL(1)), 256);
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(B_PREAD(x, 0)), 1);
            mbar_init(bar(B_PREAD(x, 1)), 1);
            mbar_init(bar(B_OFINAL(x)), 1);
        }
        mbar_init(bar(B_MMAFIN), 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == kWarpMma) {
        tmem_alloc(sb + C::kOffMisc, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == kWarpTma) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && n_max > 0) {
            uint32_t pend_mask = 0, pend_par = 0;
            mbar_arrive_expect_tx(bar(B_QFULL), kFwdTilesPerCta * C::kQBytes + C::kTileBytes);
            for (int x = 0; x < kFwdTilesPerCta; ++x)
                for (int b = 0; b < C::kBlocks; ++b)
                    tma_load_3d(sb + C::kOffQ + x * C::kQBytes + b * C::kQBlockBytes, &tmQ, b * 64,
                                q0 + x * kFwdBr, bh, bar(B_QFULL));
            for (int b = 0; b < C::kBlocks; ++b)
                tma_load_3d(sb + C::kOffK0 + b * C::kKVBlockBytes, &tmK, b * 64, 0, bh, bar(B_QFULL));
            for (int j = 0; j < n_max; ++j) {
                // stage j % kStages: V_j, then K_{j+1} (absent on the last step)
                const int s = j % C::kStages;
                const uint32_t it = (uint32_t)(j / C::kStages);
                if (!mbar_wait_bounded(bar(B_EMPTY(s)), (it & 1u) ^ 1u, abort_flag, status)) break;
                const bool next = j + 1 < n_max;
                mbar_arrive_expect_tx(bar(B_FULL(s)), next ? 2 * C::kTileBytes : C::kTileBytes);
                const uint32_t dst = sb + C::kOffRing + s * C::kStageBytes;
                for (int b = 0; b < C::kBlocks; ++b)
                    tma_load_3d(dst + b * C::kKVBlockBytes, &tmV, b * 64, j * kFwdBc, bh, bar(B_FULL(s)));
                if (next)
                    for (int b = 0; b < C::kBlocks; ++b)
                        tma_load_3d(dst + C::kTileBytes + b * C::kKVBlockBytes, &tmK, b * 64, (j + 1) * kFwdBc, bh,
                                    bar(B_FULL(s)));
                pend_mask |= 1u << s;
                pend_par = (pend_par & ~(1u << s)) | ((it & 1u) << s);
            }
            // Every load issued must land before the CTA may exit.
            volatile int no_abort = 0;
            mbar_wait_bounded(bar(B_QFULL), 0, &no_abort, status);
            for (int s = 0; s < C::kStages; ++s)
                if (pend_mask & (1u << s)) mbar_wait_bounded(bar(B_FULL(s)), (pend_par >> s) & 1u, &no_abort, status);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n_max > 0) {
            constexpr uint32_t idesc_qk = idesc_f16(128, kFwdBc, BF16, false);
            constexpr uint32_t idesc_pv = idesc_f16(128, D, BF16, true);
            // Descriptors are built once; per instruction only the address field of the
            // low word moves (by a compile-time offset plus the stage offset).
            constexpr uint32_t hi = sdesc_hi_sw128(1024);                        // 8 rows x 128 B per core group
            const uint32_t q_lo = sdesc_lo(sb + C::kOffQ, 16);                   // K-major: LBO unused
            const uint32_t k0_lo = sdesc_lo(sb + C::kOffK0, 16);
            const uint32_t ring_k_lo = sdesc_lo(sb + C::kOffRing + C::kTileBytes, 16);
            const uint32_t ring_v_lo = sdesc_lo(sb + C::kOffRing, C::kKVBlockBytes);  // MN-major: LBO = 64-col block
            // S_X = Q_X K^T for the K tile whose descriptor low word is k_lo: K-major A and
            // B, N = 64 keys, 16 of the d columns per instruction.
            auto issue_s = [&](int x, uint32_t k_lo) {
                const uint32_t qx_lo = q_lo + x * (C::kQBytes >> 4);
                const uint32_t d_s = tmem + C::tmem_s(x);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off_q = ((k >> 2) * C::kQBlockBytes + (k & 3) * 32) >> 4;
                    const uint32_t off_k = ((k >> 2) * C::kKVBlockBytes + (k & 3) * 32) >> 4;
                    umma_ss_w(d_s, qx_lo + off_q, hi, k_lo + off_k, hi, idesc_qk, k > 0 ? 1u : 0u);
                }
            };
            // O_X += P_X(j) V_j: P from TMEM buffer j % 2 (the remainder, on masked steps,
            // from the other buffer), V as an MN-major operand, 16 keys per instruction.
            auto issue_pv = [&](int x, int j, uint32_t vj_lo) {
                const uint32_t d_o = tmem + C::tmem_o(x);
                const int b = j & 1;
#pragma unroll
                for (int k = 0; k < kFwdBc / 16; ++k)
                    umma_ts_w(d_o, tmem + C::tmem_p(x, b) + 8 * k, vj_lo + ((k * 2048) >> 4), hi, idesc_pv,
                              (j > 0 || k > 0) ? 1u : 0u);
                umma_commit(bar(B_PREAD(x, b)));
                if (fwd_tile_needs_mask(j, q0 + x * kFwdBr, Nq, Nk, causal)) {
#pragma unroll
                    for (int k = 0; k < kFwdBc / 16; ++k)
                        umma_ts_w(d_o, tmem + C::tmem_p(x, b ^ 1) + 8 * k, vj_lo + ((k * 2048) >> 4), hi, idesc_pv, 1u);
                    umma_commit(bar(B_PREAD(x, b ^ 1)));
                }
                if (j == (x == 0 ? nA : nB) - 1) umma_commit(bar(B_OFINAL(x)));
            };
            bool ok = mbar_wait_bounded(bar(B_QFULL), 0, abort_flag, status);
            if (ok) {
                tc_fence_after();
                if (nA > 0) issue_s(0, k0_lo);
                if (nB > 0) issue_s(1, k0_lo);
                umma_commit(bar(B_SFULL));
            }
            for (int j = 0; ok && j < n_max; ++j) {
                const int s = j % C::kStages;
                const uint32_t stage_off = s * (C::kStageBytes >> 4);
                ok = mbar_wait_bounded(bar(B_FULL(s)), (uint32_t)(j / C::kStages) & 1u, abort_flag, status);
                if (!ok) break;
                // Next scores first: S(j+1) may overwrite S once both tiles have read S(j).
                if (j + 1 < n_max) {
                    ok = mbar_wait_bounded(bar(B_SFREE), (uint32_t)j & 1u, abort_flag, status);
                    if (!ok) break;
                    tc_fence_after();
                    if (j + 1 < nA) issue_s(0, ring_k_lo + stage_off);
                    if (j + 1 < nB) issue_s(1, ring_k_lo + stage_off);
                    umma_commit(bar(B_SFULL));
                }
                ok = mbar_wait_bounded(bar(B_PFULL(j & 1)), (uint32_t)(j >> 1) & 1u, abort_flag, status);
                if (!ok) break;
                tc_fence_after();
                if (j < nA) issue_pv(0, j, ring_v_lo + stage_off);
                if (j < nB) issue_pv(1, j, ring_v_lo + stage_off);
                umma_commit(bar(B_EMPTY(s)));
            }
            // Tensor memory may be freed only after every issued MMA completed.
            umma_commit(bar(B_MMAFIN));
            volatile int no_abort = 0;
            mbar_wait_bounded(bar(B_MMAFIN), 0, &no_abort, status);
        }
    } else {
        // ------------------------------------------------------------ softmax / correction / epilogue
        const int x = warp >> 2;       // Q tile of this warp
        const int quarter = warp & 3;  // TMEM lanes [32*quarter, 32*quarter+32) belong to this warp
        const int qx = q0 + x * kFwdBr;
        const int i = qx + quarter * 32 + lane;
        const int n_tiles = x == 0 ? nA : nB;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t s_addr = lane_base + C::tmem_s(x);
        const uint32_t o_addr = lane_base + C::tmem_o(x);
        const int lim = causal ? min(i + (Nk - Nq), Nk - 1) : Nk - 1;  // last key row i may see
        const float sl2 = args.scale_log2;
        float m = -INFINITY;  // running (possibly stale) max of scale*log2(e)*s
        float l = 0.f;        // running sum of 2^(scale*log2(e)*s - m)
        int reads0 = 0, reads1 = 0;  // MMA groups issued so far that read P_X[0] / P_X[1]
        // Wait until every MMA group that read P_X[b] so far has completed.
        auto wait_p_free = [&](int b) -> bool {
            const int r = b ? reads1 : reads0;
            if (r == 0) return true;
            return __all_sync(0xffffffffu,
                              mbar_wait_bounded(bar(B_PREAD(x, b)), (uint32_t)(r - 1) & 1u, abort_flag, status));
        };
        bool ok = true;
        // Every step of the CTA, also those past this tile's last one: the shared
        // handshake barriers need both tiles' arrivals.
        for (int j = 0; j < n_max; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(B_SFULL), (uint32_t)j & 1u, abort_flag, status));
            if (!ok) break;
            const bool active = j < n_tiles;
            uint32_t sr[64];
            if (active) {
                tc_fence_after();
                tmem_ld_32x32b_x32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
                tmem_ld_32x32b_x32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
                tmem_wait_ld();
                tc_fence_before();
            }
            mbar_arrive(bar(B_SFREE));  // S may now be overwritten by S(j+1)
            if (active) {
                const bool masked = fwd_tile_needs_mask(j, qx, Nq, Nk, causal);
                float alpha;
                bool rescale;
                uint32_t ph[32], pl[32];
                // Two instances of the same step, so the unmasked (common) step carries
                // no predicated mask or remainder instructions.
                if (masked)
                    rescale = softmax_step<true, BF16>(sr, j * kFwdBc, lim, sl2, m, l, alpha, ph, pl);
                else
                    rescale = softmax_step<false, BF16>(sr, 0, 0, sl2, m, l, alpha, ph, pl);
                const int b = j & 1;
                // P_X[b] (and on masked steps P_X[b^1]) must no longer be read by an earlier
                // MMA group; a rescale of O_X needs every earlier group complete (the latest
                // one read P_X[b^1]).
                ok = wait_p_free(b) && ((!masked && !(rescale && j > 0)) || wait_p_free(b ^ 1));
                if (!ok) break;
                tc_fence_after();
                const uint32_t p_addr = lane_base + C::tmem_p(x, b);
                tmem_st_32x32b_x16(p_addr, *reinterpret_cast<uint32_t(*)[16]>(&ph[0]));
                tmem_st_32x32b_x16(p_addr + 16, *reinterpret_cast<uint32_t(*)[16]>(&ph[16]));
                if (masked) {
                    const uint32_t plo_addr = lane_base + C::tmem_p(x, b ^ 1);
                    tmem_st_32x32b_x16(plo_addr, *reinterpret_cast<uint32_t(*)[16]>(&pl[0]));
                    tmem_st_32x32b_x16(plo_addr + 16, *reinterpret_cast<uint32_t(*)[16]>(&pl[16]));
                }
                if (rescale && j > 0) rescale_o<D>(o_addr, alpha);  // O_X holds PV_X(0..j-1), all complete
                reads0 += (b == 0 || masked) ? 1 : 0;
                reads1 += (b == 1 || masked) ? 1 : 0;
                tmem_wait_st();
                tc_fence_before();
            }
            mbar_arrive(bar(B_PFULL(j & 1)));
        }
        if (ok && n_tiles > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(B_OFINAL(x)), 0, abort_flag, status));
            tc_fence_after();
        }
        if (ok && __any_sync(0xffffffffu, i < Nq)) {
            // Epilogue: O = O~ / l (0 for a row that saw no key), LSE = m ln2 + ln l.
            const bool valid = i < Nq;
            const float inv = (l > 0.f) ? 1.f / l : 0.f;
            typename PK::T *orow_g = reinterpret_cast<typename PK::T *>(args.o) + ((size_t)bh * Nq + i) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t ov[32];
                if (n_tiles > 0) {
                    tmem_ld_32x32b_x32(o_addr + 32 * c, ov);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] = 0u;
                }
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pk[e] = PK::pack(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
                if (valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow_g + 32 * c);
#pragma unroll
                    for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                }
            }
            if (valid && args.lse != nullptr) {
                const float m_fin = (m == -INFINITY) ? 0.f : m;
                args.lse[(size_t)bh * Nq + i] = (l > 0.f) ? m_fin * 0.69314718055994531f + logf(l) : -INFINITY;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool BF16>
static cudaError_t launch_fwd_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                                const FwdArgs &a, int BH, cudaStream_t stream) {
    using C = FwdCfg<D>;
    auto kern = fa_fwd_kernel<D, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)a.num_m, (unsigned)BH, 1);
    kern<<<grid, kFwdThreads, C::kSmemBytes, stream>>>(tq, tk, tv, a);
    return cudaGetLastError();
}

cudaError_t launch_fwd(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const FwdArgs &a, int BH, cudaStream_t stream) {
    if (d == 64) return bf16 ? launch_fwd_t<64, true>(tq, tk, tv, a, BH, stream)
                             : launch_fwd_t<64, false>(tq, tk, tv, a, BH, stream);
    return bf16 ? launch_fwd_t<128, true>(tq, tk, tv, a, BH, stream)
                : launch_fwd_t<128, false>(tq, tk, tv, a, BH, stream);
}

}  // namespace fa
