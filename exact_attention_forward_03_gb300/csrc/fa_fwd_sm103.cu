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
// Roles (warp specialisation, 5 warpgroups):
//   warps 0-7   softmax of Q tile A: warp w handles TMEM lanes (rows)
//               [32*(w%4), +32) and columns [64*h, +64) of the 128-key tile,
//               h = (w/4)%2; the two warps of a row pair exchange their partial
//               row maxima through shared memory (a 64-thread named barrier)
//   warps 8-15  the same for Q tile B
//   warp 16     TMA producer: both Q tiles once, then K_0, V_0, K_1, V_1, ...
//               through a ring of shared-memory slots (full/empty mbarriers)
//   warp 17     owns tensor memory; one lane issues every tcgen05.mma
//   warps 18-19 idle (they complete the fifth warpgroup)
// Splitting a row over two warps puts two softmax warps of each tile on every
// SM sub-partition, so the exp2 pipe stays fed and a tile's softmax takes half
// as long.  The launch gives 96 registers per thread; the fifth warpgroup
// drops to 64 and the softmax warpgroups rise to 104 (64 + 4 * 104 = 5 * 96).
//
// The two Q tiles ping-pong on the tensor core: while the softmax warps of one
// tile work on S_j, the tensor core runs O += P_j V_j and S_{j+1} = Q K_{j+1}^T
// of the other tile, so exp2 and the rescale stay off the tensor pipe's path.
// MMA issue order per K/V step j:  PV_A(j), S_A(j+1), PV_B(j), S_B(j+1).
//
// Tensor memory (512 columns): S_A [0,128), S_B [128,256), O_A [256,256+d),
// O_B [256+d,256+2d).  P_X overwrites the first 64 columns of S_X as 16-bit
// pairs once the softmax threads hold their S values in registers; on tiles
// that need a mask the 16-bit remainder P - P_hi goes to the next 64 columns
// and is multiplied into O as well (rows near the diagonal see few keys, so
// one 16-bit rounding of their few large weights would dominate their error).
// tcgen05.mma operations of one thread run in issue order, so S_X(j+1) writes
// S_X only after PV_X(j) has read P_X(j); and the commit that signals S_X(j+1)
// also covers PV_X(j), so the softmax may rescale O_X as soon as S_X(j+1) is ready.
//
// The rescale of O by alpha = 2^(m_old - m_new) is done only when the row max
// of some row in the warp grew by more than 2^8: otherwise m stays and p may
// reach 2^8, which changes nothing in exact arithmetic (O and l share the same
// stale max) and keeps fp16/bf16/fp32 far from overflow.
//
// Every mbarrier wait is bounded (%globaltimer); on expiry the CTA records
// the timeout in the status word, stops issuing work, waits (bounded) for its
// in-flight TMA loads and MMAs, frees tensor memory and exits.  The two warps
// of a row pair AND their wait results at every pair barrier, so both leave
// together.
#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {

constexpr int kFwdThreads = 640;
constexpr int kWarpTma = 16, kWarpMma = 17;
constexpr uint32_t kRegsSoftmax = 104;
constexpr uint32_t kRegsOther = 64;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct FwdCfg {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int kStages = (D == 128) ? 4 : 8;
    static constexpr int kBlocks = D / 64;               // 128-byte swizzle blocks per row
    static constexpr int kQBlockBytes = kFwdBr * 128;    // one 64-column block of a Q tile
    static constexpr int kKVBlockBytes = kFwdBc * 128;   // one 64-column block of a K/V tile
    static constexpr int kQBytes = kFwdBr * D * 2;       // one Q tile
    static constexpr int kTileBytes = kFwdBc * D * 2;    // one K or V tile
    static constexpr int kOffQ = 0;                      // Q_A, then Q_B
    static constexpr int kOffRing = kFwdTilesPerCta * kQBytes;
    static constexpr int kOffBar = kOffRing + kStages * kTileBytes;
    // barriers: q_full, full[S], empty[S], s_full[2], p_full[2], o_final[2], mma_fin
    static constexpr int kNumBars = 1 + 2 * kStages + 2 + 2 + 2 + 1;
    static constexpr int kOffRed = kOffBar + kNumBars * 8;      // float red[2 parity][2 tiles][2 halves][128 rows]
    static constexpr int kOffMisc = kOffRed + 2 * 2 * 2 * 128 * 4;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack to align the base to 1024
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
    static constexpr uint32_t kTmemCols = 512;
    __device__ static constexpr uint32_t tmem_s(int x) { return x == 0 ? 0u : 128u; }
    __device__ static constexpr uint32_t tmem_o(int x) { return x == 0 ? 256u : 256u + D; }
};

// Tile j needs element masks when it crosses the ragged end of K or, under
// causal masking, holds a key beyond the first row's last visible key.
__device__ __forceinline__ bool fwd_tile_needs_mask(int j, int q0, int Nq, int Nk, int causal) {
    const int last_key = (j + 1) * kFwdBc - 1;
    return (last_key >= Nk) || (causal && last_key > q0 + (Nk - Nq));
}

// K/V tiles that Q rows [q0, q0+128) must visit (0 when the tile holds no row).
__device__ __forceinline__ int fwd_tile_count(int q0, int Nq, int Nk, int causal) {
    if (q0 >= Nq) return 0;
    int kv_end = Nk;
    if (causal) kv_end = min(Nk, min(q0 + kFwdBr, Nq) + (Nk - Nq));
    return kv_end > 0 ? (kv_end + kFwdBc - 1) / kFwdBc : 0;
}

// Per-thread state of one softmax thread: one row, 64 of the tile's columns.
struct RowState {
    float m;  // running (possibly stale) max of scale*log2(e)*s over the whole row
    float l;  // this thread's share of the running sum of 2^(scale*log2(e)*s - m)
};

// Exponentials of one 32-column chunk of S: p = 2^(s*c - m_d) for the 32 values
// in `sr`, their sum added to `rs2`, and the packed 16-bit P (and on masked
// tiles the 16-bit remainder) stored to TMEM at `p_addr` (and `plo_addr`).
template <bool MASKED, bool BF16>
__device__ __forceinline__ void exp_chunk(const uint32_t (&sr)[32], uint64_t scale2, uint64_t shift2,
                                          uint64_t (&rs2)[2], uint32_t p_addr, uint32_t plo_addr) {
    using PK = Pack<BF16>;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        uint32_t ph[8], pl[8];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
            const int col = 16 * c + e;
            const float2 xa = f2_split(ffma2(f2_make(__uint_as_float(sr[col]), __uint_as_float(sr[col + 1])), scale2, shift2));
            const float p0 = ex2_approx(xa.x);
            const float p1 = ex2_approx(xa.y);
            rs2[(e >> 1) & 1] = fadd2(rs2[(e >> 1) & 1], f2_make(p0, p1));
            ph[e >> 1] = PK::pack(p0, p1);
            if (MASKED) {
                const float2 hf = PK::unpack(ph[e >> 1]);
                pl[e >> 1] = PK::pack(p0 - hf.x, p1 - hf.y);
            }
        }
        tmem_st_32x32b_x8(p_addr + 8 * c, ph);
        if (MASKED) tmem_st_32x32b_x8(plo_addr + 8 * c, pl);
    }
}

template <bool MASKED>
__device__ __forceinline__ void mask_chunk(uint32_t (&sr)[32], int c0, int lim) {
    if (MASKED) {
#pragma unroll
        for (int c = 0; c < 32; ++c)
            if (c0 + c > lim) sr[c] = __float_as_uint(-INFINITY);
    }
}

__device__ __forceinline__ float max_chunk(const uint32_t (&sr)[32]) {
    float mx[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) mx[e] = fmax3(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1]), -INFINITY);
#pragma unroll
    for (int c = 8; c < 32; c += 2) mx[(c >> 1) & 3] = fmax3(mx[(c >> 1) & 3], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
    return fmaxf(fmax3(mx[0], mx[1], mx[2]), mx[3]);
}

// One online-softmax step for this warp's 64 columns of the S row (TMEM at
// `s_addr`): optional causal/tail mask, partial max exchanged with the partner
// warp, (conditional) max update, p = 2^(s*c - m), this half's row sum, and P
// written back as 16-bit pairs into this half's own TMEM columns.  Only one
// 32-column chunk of S is held in registers at a time: chunk 0 is read for its
// max, chunk 1 is read and turned into P, then chunk 0 is read again.  Layout of
// the half's 64 columns afterwards: P of chunk 0 at [0,16), its remainder at
// [16,32), the remainder of chunk 1 at [32,48), P of chunk 1 at [48,64) (the
// remainders only on masked tiles).  Returns false if the pair must abort;
// otherwise `rescale` says whether the warp moved its max and `alpha` is the
// factor O and l are scaled by.
template <bool MASKED, bool BF16>
__device__ __forceinline__ bool softmax_half(uint32_t s_addr, int c0, int lim, float sl2, RowState &st, float &alpha,
                                             bool &rescale, float *red_mine, const float *red_other, int pair_bar,
                                             bool ok) {
    uint32_t sr[32];
    float mine = -INFINITY;
    if (ok) {
        tmem_ld_32x32b_x32(s_addr, sr);
        tmem_wait_ld();
        mask_chunk<MASKED>(sr, c0, lim);
        mine = max_chunk(sr);
        tmem_ld_32x32b_x32(s_addr + 32, sr);
        tmem_wait_ld();
        mask_chunk<MASKED>(sr, c0 + 32, lim);
        mine = fmaxf(mine, max_chunk(sr));
    }
    *red_mine = mine;
    if (!named_bar_and(pair_bar, 64, ok)) return false;
    const float mt = fmaxf(mine, *red_other);
    const float m_cand = fmaxf(st.m, mt * sl2);
    rescale = __any_sync(0xffffffffu, m_cand > st.m + kRescaleThreshold);
    alpha = 1.f;
    if (rescale) {
        const float m_new_d = (m_cand == -INFINITY) ? 0.f : m_cand;  // never subtract -inf from -inf
        alpha = ex2_approx(st.m - m_new_d);
        st.m = m_cand;
    }
    const float m_d = (st.m == -INFINITY) ? 0.f : st.m;
    const uint64_t scale2 = f2_make(sl2, sl2);
    const uint64_t shift2 = f2_make(-m_d, -m_d);
    uint64_t rs2[2] = {f2_make(0.f, 0.f), f2_make(0.f, 0.f)};
    exp_chunk<MASKED, BF16>(sr, scale2, shift2, rs2, s_addr + 48, s_addr + 32);  // chunk 1, still in registers
    tmem_ld_32x32b_x32(s_addr, sr);                                               // chunk 0 again
    tmem_wait_ld();
    mask_chunk<MASKED>(sr, c0, lim);
    exp_chunk<MASKED, BF16>(sr, scale2, shift2, rs2, s_addr, s_addr + 16);
    const float2 r0 = f2_split(rs2[0]), r1 = f2_split(rs2[1]);
    st.l = st.l * alpha + ((r0.x + r0.y) + (r1.x + r1.y));
    return true;
}

template <bool BF16>
__device__ __noinline__ bool softmax_half_masked(uint32_t s_addr, int c0, int lim, float sl2, RowState &st, float &alpha,
                                                 bool &rescale, float *red_mine, const float *red_other, int pair_bar, bool ok) {
    return softmax_half<true, BF16>(s_addr, c0, lim, sl2, st, alpha, rescale, red_mine, red_other, pair_bar, ok);
}

// O_X (this warp's kOHalf columns of 32 rows) *= alpha, 16 columns at a time.
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
    auto B_SFULL = [](int x) { return 1 + 2 * C::kStages + x; };
    auto B_PFULL = [](int x) { return 3 + 2 * C::kStages + x; };
    auto B_OFINAL = [](int x) { return 5 + 2 * C::kStages + x; };
    constexpr int B_MMAFIN = 7 + 2 * C::kStages;
    volatile uint32_t *tmem_holder = reinterpret_cast<volatile uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
    int *status = args.status;

    if (threadIdx.x == 0) {
        mbar_init(bar(B_QFULL), 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar(B_FULL(s)), 1);
            mbar_init(bar(B_EMPTY(s)), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(B_SFULL(x)), 1);
            mbar_init(bar(B_PFULL(x)), 256);
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

    if (warp >= 16) {
        regs_decrease<kRegsOther>();
        if (warp == kWarpTma && lane == 0 && n_max > 0) {
            // ------------------------------------------------------------ TMA producer
            uint32_t pend_mask = 0, pend_par = 0;
            mbar_arrive_expect_tx(bar(B_QFULL), kFwdTilesPerCta * C::kQBytes);
            for (int x = 0; x < kFwdTilesPerCta; ++x)
                for (int b = 0; b < C::kBlocks; ++b)
                    tma_load_3d(sb + C::kOffQ + x * C::kQBytes + b * C::kQBlockBytes, &tmQ, b * 64,
                                q0 + x * kFwdBr, bh, bar(B_QFULL));
            for (int t = 0; t < 2 * n_max; ++t) {
                const int s = t % C::kStages;
                const uint32_t it = (uint32_t)(t / C::kStages);
                if (!mbar_wait_bounded(bar(B_EMPTY(s)), (it & 1u) ^ 1u, abort_flag, status)) break;
                mbar_arrive_expect_tx(bar(B_FULL(s)), C::kTileBytes);
                const CUtensorMap *map = (t & 1) ? &tmV : &tmK;
                const int y = (t >> 1) * kFwdBc;
                const uint32_t dst = sb + C::kOffRing + s * C::kTileBytes;
                for (int b = 0; b < C::kBlocks; ++b)
                    tma_load_3d(dst + b * C::kKVBlockBytes, map, b * 64, y, bh, bar(B_FULL(s)));
                pend_mask |= 1u << s;
                pend_par = (pend_par & ~(1u << s)) | ((it & 1u) << s);
            }
            // Every load issued must land before the CTA may exit.
            volatile int no_abort = 0;
            mbar_wait_bounded(bar(B_QFULL), 0, &no_abort, status);
            for (int s = 0; s < C::kStages; ++s)
                if (pend_mask & (1u << s)) mbar_wait_bounded(bar(B_FULL(s)), (pend_par >> s) & 1u, &no_abort, status);
        } else if (warp == kWarpMma && lane == 0 && n_max > 0) {
            // ------------------------------------------------------------ MMA issuer
            constexpr uint32_t idesc_qk = idesc_f16(128, kFwdBc, BF16, false);
            constexpr uint32_t idesc_pv = idesc_f16(128, D, BF16, true);
            const int n_x[2] = {nA, nB};
            auto slot_of = [](int t) { return t % C::kStages; };
            auto par_of = [](int t) { return (uint32_t)(t / C::kStages) & 1u; };
            // Descriptors are built once; per instruction only the address field of the
            // low word moves (by a compile-time offset plus the slot offset).
            constexpr uint32_t hi = sdesc_hi_sw128(1024);                        // 8 rows x 128 B per core group
            const uint32_t q_lo = sdesc_lo(sb + C::kOffQ, 16);                   // K-major: LBO unused
            const uint32_t k_lo = sdesc_lo(sb + C::kOffRing, 16);
            const uint32_t v_lo = sdesc_lo(sb + C::kOffRing, C::kKVBlockBytes);  // MN-major: LBO = 64-col block
            // S_X(j) = Q_X K_j^T: K-major A and B, 16 of the d columns per instruction.
            auto issue_s = [&](int x, int j) {
                const uint32_t qx_lo = q_lo + x * (C::kQBytes >> 4);
                const uint32_t kj_lo = k_lo + slot_of(2 * j) * (C::kTileBytes >> 4);
                const uint32_t d_s = tmem + C::tmem_s(x);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off_q = ((k >> 2) * C::kQBlockBytes + (k & 3) * 32) >> 4;
                    const uint32_t off_k = ((k >> 2) * C::kKVBlockBytes + (k & 3) * 32) >> 4;
                    umma_ss_w(d_s, qx_lo + off_q, hi, kj_lo + off_k, hi, idesc_qk, k > 0 ? 1u : 0u);
                }
                umma_commit(bar(B_SFULL(x)));
            };
            // O_X += P_X(j) V_j: P from TMEM, V as an MN-major operand, 16 keys per instruction.
            // Keys [64h + 32c, +32) of P sit at columns 64h + 32c + {0, 16} (P, remainder)
            // for chunk c = 0 and 64h + {48, 32} for chunk c = 1 (see softmax_half).
            auto p_col = [](int k) { return (uint32_t)(64 * (k >> 2) + 8 * (k & 3) + ((k & 2) ? 32 : 0)); };
            auto plo_col = [](int k) { return (uint32_t)(64 * (k >> 2) + 8 * (k & 3) + 16); };
            auto issue_pv = [&](int x, int j) {
                const uint32_t vj_lo = v_lo + slot_of(2 * j + 1) * (C::kTileBytes >> 4);
                const uint32_t d_o = tmem + C::tmem_o(x);
                const uint32_t p_t = tmem + C::tmem_s(x);
#pragma unroll
                for (int k = 0; k < kFwdBc / 16; ++k)
                    umma_ts_w(d_o, p_t + p_col(k), vj_lo + ((k * 2048) >> 4), hi, idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
                if (fwd_tile_needs_mask(j, q0 + x * kFwdBr, Nq, Nk, causal)) {
#pragma unroll
                    for (int k = 0; k < kFwdBc / 16; ++k)
                        umma_ts_w(d_o, p_t + plo_col(k), vj_lo + ((k * 2048) >> 4), hi, idesc_pv, 1u);
                }
                if (j == n_x[x] - 1) umma_commit(bar(B_OFINAL(x)));
            };
            bool ok = mbar_wait_bounded(bar(B_QFULL), 0, abort_flag, status) &&
                      mbar_wait_bounded(bar(B_FULL(slot_of(0))), par_of(0), abort_flag, status);
            if (ok) {
                tc_fence_after();
                if (nA > 0) issue_s(0, 0);
                if (nB > 0) issue_s(1, 0);
                umma_commit(bar(B_EMPTY(slot_of(0))));
            }
            for (int j = 0; ok && j < n_max; ++j) {
                const bool next = j + 1 < n_max;
                bool v_ready = false, k_ready = false;  // V_j and K_{j+1} checked once per step
                for (int x = 0; ok && x < 2; ++x) {
                    if (j < n_x[x]) {
                        // P_X(j) first: it is the wait most likely to block.
                        if (!mbar_wait_bounded(bar(B_PFULL(x)), (uint32_t)j & 1u, abort_flag, status) ||
                            (!v_ready &&
                             !mbar_wait_bounded(bar(B_FULL(slot_of(2 * j + 1))), par_of(2 * j + 1), abort_flag, status))) {
                            ok = false;
                            break;
                        }
                        v_ready = true;
                        tc_fence_after();
                        issue_pv(x, j);
                    }
                    if (j + 1 < n_x[x]) {
                        if (!k_ready &&
                            !mbar_wait_bounded(bar(B_FULL(slot_of(2 * j + 2))), par_of(2 * j + 2), abort_flag, status)) {
                            ok = false;
                            break;
                        }
                        k_ready = true;
                        tc_fence_after();
                        issue_s(x, j + 1);
                    }
                }
                if (!ok) break;
                umma_commit(bar(B_EMPTY(slot_of(2 * j + 1))));
                if (next) umma_commit(bar(B_EMPTY(slot_of(2 * j + 2))));
            }
            // Tensor memory may be freed only after every issued MMA completed.
            umma_commit(bar(B_MMAFIN));
            volatile int no_abort = 0;
            mbar_wait_bounded(bar(B_MMAFIN), 0, &no_abort, status);
        }
    } else {
        // ------------------------------------------------------------ softmax / correction / epilogue
        regs_increase<kRegsSoftmax>();
        const int x = warp >> 3;          // Q tile of this warp
        const int h = (warp >> 2) & 1;    // column half of the 128-key tile
        const int quarter = warp & 3;     // TMEM lanes [32*quarter, 32*quarter+32) belong to this warp
        const int r = quarter * 32 + lane;
        const int qx = q0 + x * kFwdBr;
        const int i = qx + r;
        const int n_tiles = x == 0 ? nA : nB;
        const int pair_bar = 1 + x * 4 + quarter;  // named barrier shared with the other column half
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t s_addr = lane_base + C::tmem_s(x) + 64 * h;          // this half's S columns
        constexpr int kOHalf = D / 2;                                          // O columns owned by this warp
        const uint32_t o_addr = lane_base + C::tmem_o(x) + kOHalf * h;
        float *red = reinterpret_cast<float *>(smem + C::kOffRed);
        auto red_at = [&](int parity, int half) { return red + ((parity * 2 + x) * 2 + half) * 128 + r; };
        const int lim = causal ? min(i + (Nk - Nq), Nk - 1) : Nk - 1;  // last key row i may see
        const float sl2 = args.scale_log2;
        RowState st{-INFINITY, 0.f};
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(B_SFULL(x)), (uint32_t)j & 1u, abort_flag, status));
            if (ok) tc_fence_after();
            const bool masked = fwd_tile_needs_mask(j, qx, Nq, Nk, causal);
            float alpha;
            bool rescale;
            float *mine = red_at(j & 1, h);
            const float *other = red_at(j & 1, h ^ 1);
            // Two instances of the same step, so the unmasked (common) tile carries
            // no predicated mask or remainder instructions.
            if (masked)
                ok = softmax_half_masked<BF16>(s_addr, j * kFwdBc + 64 * h, lim, sl2, st, alpha, rescale, mine, other,
                                              pair_bar, ok);
            else
                ok = softmax_half<false, BF16>(s_addr, 0, 0, sl2, st, alpha, rescale, mine, other, pair_bar, ok);
            if (!ok) break;
            if (rescale && j > 0) rescale_o<kOHalf>(o_addr, alpha);  // O_X holds PV_X(0..j-1), all complete
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(B_PFULL(x)));
        }
        if (ok && n_tiles > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(B_OFINAL(x)), 0, abort_flag, status));
            tc_fence_after();
        }
        // Row sum: the two column halves add their shares.  The first barrier keeps
        // this write of parity buffer 0 behind the partner's last read of it.
        named_bar_sync(pair_bar, 64);
        *red_at(0, h) = st.l;
        ok = named_bar_and(pair_bar, 64, ok);
        const float l = st.l + *red_at(0, h ^ 1);
        if (ok && __any_sync(0xffffffffu, i < Nq)) {
            // Epilogue: O = O~ / l (0 for a row that saw no key), LSE = m ln2 + ln l.
            const bool valid = i < Nq;
            const float inv = (l > 0.f) ? 1.f / l : 0.f;
            typename PK::T *orow_g =
                reinterpret_cast<typename PK::T *>(args.o) + ((size_t)bh * Nq + i) * D + kOHalf * h;
#pragma unroll
            for (int c = 0; c < kOHalf / 32; ++c) {
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
            if (valid && h == 0 && args.lse != nullptr) {
                const float m_fin = (st.m == -INFINITY) ? 0.f : st.m;
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
