// fa_fwd_sm103.cu -- fused exact attention forward on sm_103a tensor cores.
//
// One CTA computes one 128-row Q tile of one (batch, head):
//   O_i = sum_j softmax_j(scale * q_i . k_j + mask) v_j,  LSE_i = m_i + ln l_i
// following the FlashAttention-2 forward ("6.2 FlashAttention V2 explained",
// §6): the Q tile stays on chip, K/V tiles stream past it, a running row max m
// and row sum l are kept per row, the accumulator is rescaled by
// exp(m_old - m_new) and divided by l once at the end (§3.2; "02 · FA2", §1).
// Causal masking visits only K/V tiles up to the diagonal and masks
// element-wise only on tiles that straddle it or the ragged Nk tail (§5.3;
// "02 · FA2", §4).
//
// Roles (warp specialisation, 8 warps):
//   warps 0-3  softmax: one thread per query row (TMEM lane = row), the whole
//              128-key row of S in registers; then the epilogue
//   warp 4     TMA producer: the Q tile once, then K_0, K_1, K_2, V_0, K_3,
//              V_1, K_4, ... into two rings of shared-memory slots, one for K
//              tiles and one for V tiles (full/empty mbarriers per slot).  Its
//              lane initialises the barriers and issues Q and K_0..K_2 before
//              the CTA-wide sync on the tensor-memory allocation.
//   warp 5     owns tensor memory; one lane issues O += P(j) V_j for every j
//   warp 6     one lane issues S(t) = Q K_t^T for every t
//   warp 7     idle
//
// Tensor memory (512 columns; see the paired form below): three score buffers S[0..2] = [0,128),
// [128,256), [256,384), and O = [384, 384+d).  Tile j's scores go to
// S[j % 3].  Once a softmax thread holds its row of S(j) in registers it
// writes P(j) as 16-bit pairs over the first 64 columns of that buffer (and,
// on tiles that need a mask, the 16-bit remainder P - P_head over the next 64:
// rows near the diagonal see few keys, so one 16-bit rounding of their few
// large weights would otherwise dominate their error; both parts are
// multiplied into O).
//
// S(t) may overwrite S[t % 3] once PV(t-3) has read P(t-3) from it, so the
// scores run up to three tiles ahead of the softmax, which goes from one tile
// to the next without waiting for the tensor core.  The two MMA streams come
// from two threads: the PV stream waits for each P, the S stream runs ahead
// and fills the tensor core whenever the PV stream waits or does its
// bookkeeping.  Only the softmax is on the critical path.
//
// The running max m only keeps p in range: O and l share it, so a stale m
// changes nothing in exact arithmetic.  The exact row max is taken on a row's
// first tile and on masked tiles, where m moves (and O is rescaled by
// alpha = 2^(m_old - m_new)) only if the max grew by more than 2^8; on the
// other tiles the exponentials are taken against the current m at once and the
// tile's row sum checks them (see softmax_tile).  A rescale at tile j waits for
// PV(j-1) to complete.
//
// Barrier phases: S(t), P(j) and "PV(j) done" each use three barriers indexed
// by tile mod 3, so that no waiter can fall two phases behind on the barrier
// it waits on (every pair of producer and consumer is at most two tiles apart).
//
// Epilogue: O = O~ / l and LSE per row; the 16-bit O rows are staged in the
// freed K ring slot 0 in the Q/K tile layout, one 64-column block at a time, and
// each block leaves as a TMA store as soon as all its rows are staged, reading
// shared memory while the next block is packed (a packed batch's partial last
// row block of a sequence is stored row by row instead, since its box would
// overlap the next sequence's rows).
//
// Paired form (d = 64, grids of a few waves with short rows): two CTAs share an
// SM.  Each takes 256 tensor-memory columns (one score buffer S[0] = [0,128) and
// O = [128, 128+d)) and about 81 KB of shared memory (two-slot K and V rings),
// and is launched at 128 registers per thread; the softmax warpgroup raises its
// share to 208 and the producer/issuer warpgroup lowers its to 48 (setmaxnreg).
// With one score buffer S(t+1) waits for PV(t), so each CTA's tiles go
// S -> softmax -> PV one after another; the other CTA's chain, set-up and
// epilogue fill the gaps.  The barriers and phases are those of the three-buffer
// form with the buffer count as the modulus.
//
// Every mbarrier wait is bounded (%globaltimer); on expiry the CTA records
// the timeout in the status word, stops issuing work, waits (bounded) for its
// in-flight TMA loads and MMAs, frees tensor memory and exits.
#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {

constexpr int kFwdThreads = 256;
constexpr int kWarpTma = 4, kWarpPv = 5, kWarpS = 6;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kRowSumLimit = 32768.0f;   // 2^15

// PAIR: two CTAs share an SM (d = 64 only), each with one score buffer and
// 256 tensor-memory columns; the two CTAs' S -> softmax -> PV chains interleave
// on the SM, and one CTA's set-up and epilogue overlap the other's tile loop.
template <int D, bool PAIR = false>
struct FwdCfg {
    static_assert(D == 64 || D == 128, "head dim");
    static_assert(!PAIR || D == 64, "two CTAs per SM only at d = 64");
    static constexpr int kBlocks = D / 64;               // 128-byte swizzle blocks per row
    static constexpr int kQBlockBytes = kFwdBr * 128;    // one 64-column block of the Q tile
    static constexpr int kKVBlockBytes = kFwdBc * 128;   // one 64-column block of a K/V tile
    static constexpr int kQBytes = kFwdBr * D * 2;       // the Q tile
    static constexpr int kTileBytes = kFwdBc * D * 2;    // one K or V tile
    static constexpr int kStages = PAIR ? 2 : (D == 128) ? 3 : 6;  // slots per ring (one K ring, one V ring)
    static constexpr int kSBuf = PAIR ? 1 : 3;           // score buffers in tensor memory
    static constexpr int kAhead = PAIR ? 2 : 3;          // K tiles loaded before the first V tile
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kQBytes;
    static constexpr int kOffV = kOffK + kStages * kTileBytes;
    static constexpr int kOffBar = kOffV + kStages * kTileBytes;
    // barriers: q_full, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[3], p_full[3],
    // pv_done[3], o_final, mma_fin[2]
    static constexpr int kNumBars = 1 + 4 * kStages + 9 + 1 + 2;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack to align the base to 1024
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
    static_assert(!PAIR || 2 * (kSmemBytes + 1024) <= 233472, "two CTAs per SM");
    static constexpr uint32_t kTmemCols = PAIR ? 256 : 512;
    __device__ static constexpr uint32_t tmem_s(int b) { return 128u * b; }
    static constexpr uint32_t kTmemO = 128u * kSBuf;
    static_assert(kTmemO + D <= kTmemCols, "tensor memory");
};

// K/V tile j needs element masks when it crosses the ragged end of K or, under
// causal masking, holds a key beyond the first row's last visible key:
//   (j+1)*Bc - 1 >= Nk  or  (causal and (j+1)*Bc - 1 > q0 + Nk - Nq).
// Both conditions are monotone in j; this returns the first tile that meets
// either, so tile j needs masks exactly when j >= fwd_first_masked_tile(...).
__device__ __forceinline__ int fwd_first_masked_tile(int q0, int Nq, int Nk, int causal) {
    const int j_tail = Nk / kFwdBc;
    if (!causal) return j_tail;
    const int d1 = q0 + (Nk - Nq) + 1;
    return min(j_tail, d1 <= 0 ? 0 : d1 / kFwdBc);
}

// K/V tiles that Q rows [q0, q0+128) must visit (0 when the tile holds no row).
__device__ __forceinline__ int fwd_tile_count(int q0, int Nq, int Nk, int causal) {
    if (q0 >= Nq) return 0;
    int kv_end = Nk;
    if (causal) kv_end = min(Nk, min(q0 + kFwdBr, Nq) + (Nk - Nq));
    return kv_end > 0 ? (kv_end + kFwdBc - 1) / kFwdBc : 0;
}

// State of one softmax thread's row after a step.
struct RowStep {
    float m;       // running (possibly stale) max of scale*log2(e)*s
    float l;       // running sum of 2^(scale*log2(e)*s - m)
    float alpha;   // factor O is to be scaled by in this step
    bool rescale;  // whether the warp moved its max in this step
};

// Largest of the row's 128 scores (fp32 bits; -inf entries count as -inf).
__device__ __forceinline__ float row_max(const uint32_t (&s)[128]) {
    float mx[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) mx[e] = fmax3(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1]), -INFINITY);
#pragma unroll
    for (int c = 16; c < 128; c += 2)
        mx[(c >> 1) & 7] = fmax3(mx[(c >> 1) & 7], __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
    return fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
}

// p = 2^(s*c - m_d) for the row's 128 scores, written as 16-bit pairs over the
// first 64 TMEM columns at s_addr (keys [16k, 16k+16) in columns [8k, 8k+8);
// on masked tiles the 16-bit remainder p - p_head over the next 64); returns
// the fp32 sum of the p.
template <bool MASKED, bool BF16>
__device__ __forceinline__ float exp_row(const uint32_t (&s)[128], uint32_t s_addr, float sl2, float m_d) {
    using PK = Pack<BF16>;
    const uint64_t scale2 = f2_make(sl2, sl2);
    const uint64_t shift2 = f2_make(-m_d, -m_d);
    uint64_t rs2[4] = {f2_make(0.f, 0.f), f2_make(0.f, 0.f), f2_make(0.f, 0.f), f2_make(0.f, 0.f)};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t ph[16], pl[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
            const int col = 32 * c + e;
            const float2 xa = f2_split(ffma2(f2_make(__uint_as_float(s[col]), __uint_as_float(s[col + 1])), scale2, shift2));
            const float p0 = ex2_approx(xa.x);
            const float p1 = ex2_approx(xa.y);
            rs2[(e >> 1) & 3] = fadd2(rs2[(e >> 1) & 3], f2_make(p0, p1));
            ph[e >> 1] = PK::pack(p0, p1);
            if (MASKED) {
                const float2 hf = PK::unpack(ph[e >> 1]);
                pl[e >> 1] = PK::pack(p0 - hf.x, p1 - hf.y);
            }
        }
        tmem_st_32x32b_x16(s_addr + 16 * c, ph);
        if (MASKED) tmem_st_32x32b_x16(s_addr + 64 + 16 * c, pl);
    }
    const float2 r0 = f2_split(fadd2(rs2[0], rs2[1])), r1 = f2_split(fadd2(rs2[2], rs2[3]));
    return (r0.x + r0.y) + (r1.x + r1.y);
}

// One online-softmax step of this thread's row over one K/V tile: S (128 fp32
// columns of TMEM at s_addr) into registers, optional causal/tail mask, the
// exponentials against the running max m, the row sum, and P over the first
// 64 columns of S (see exp_row).
//
// Any finite m gives the same O and l in exact arithmetic (O and l are both
// relative to it), so m only has to keep p within range.  The exact row max is
// taken on a row's first tile and on masked tiles (where a max that grew by
// more than 2^8 moves m and rescales O).  On the other tiles the exponentials
// are taken against the current m straight away, with no max pass, and the
// tile's row sum checks the result: when every row of the warp summed to at
// most 2^15, every p is at most 2^15 (inside fp16 and bf16) and the tile
// stands; otherwise (the scores rose well above m) the warp takes the exact
// max, moves m, and redoes the tile.
template <bool MASKED, bool BF16>
__device__ __forceinline__ RowStep softmax_tile(uint32_t s_addr, int c0, int lim, float sl2, float m, float l) {
    uint32_t s[128];
    tmem_ld_32x32b_x32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
    tmem_ld_32x32b_x32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
    tmem_ld_32x32b_x32(s_addr + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
    tmem_ld_32x32b_x32(s_addr + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
    tmem_wait_ld();
    if (MASKED) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
            if (c0 + c > lim) s[c] = __float_as_uint(-INFINITY);
    }
    RowStep r;
    r.rescale = false;
    r.alpha = 1.f;
    const bool exact = MASKED || __any_sync(0xffffffffu, m == -INFINITY);
    if (exact) {
        const float m_cand = fmaxf(m, row_max(s) * sl2);
        r.rescale = __any_sync(0xffffffffu, m_cand > m + kRescaleThreshold);
        if (r.rescale) {
            const float m_new_d = (m_cand == -INFINITY) ? 0.f : m_cand;  // never subtract -inf from -inf
            r.alpha = ex2_approx(m - m_new_d);
            m = m_cand;
        }
    }
    float sum = exp_row<MASKED, BF16>(s, s_addr, sl2, (m == -INFINITY) ? 0.f : m);
    if (!exact && __any_sync(0xffffffffu, sum > kRowSumLimit)) {
        // m is finite on every row of the warp here, and m_cand >= m.
        const float m_cand = fmaxf(m, row_max(s) * sl2);
        r.alpha = ex2_approx(m - m_cand);
        r.rescale = true;
        m = m_cand;
        sum = exp_row<false, BF16>(s, s_addr, sl2, m);
    }
    r.m = m;
    r.l = l * r.alpha + sum;
    return r;
}

// The masked step is taken about once per Q tile, so it is kept out of line to
// leave the registers and code of the common step alone.
template <bool BF16>
__device__ __noinline__ RowStep softmax_tile_masked(uint32_t s_addr, int c0, int lim, float sl2, float m, float l) {
    return softmax_tile<true, BF16>(s_addr, c0, lim, sl2, m, l);
}

// O (32 rows of this warp, kCols columns) *= alpha, 16 columns at a time.
// Rarely taken (only when a row max grows by more than 2^8).
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

// VARLEN: packed variable-length batch.  by = sequence * H + head, q, o
// are [total_q, H, d], k, v are [total_k, H_kv, d] (tensor maps indexed by column,
// head, token), lse is [H, total_q], and sequence s spans tokens
// [cu_q[s], cu_q[s+1]) of q and [cu_k[s], cu_k[s+1]) of k and v.  A key tile may
// run past its sequence's last key into the next sequence: those keys are masked
// like the ragged tail of a dense K.  Query rows past the sequence are not stored.
// Register split of the PAIR form (launched at 128 per thread so that two CTAs fit):
// the softmax warpgroup takes 208, the producer/issuer warpgroup keeps 48.
constexpr uint32_t kPairRegsLaunch = 128, kPairRegsSoftmax = 208, kPairRegsIo = 48;
static_assert(kPairRegsSoftmax + kPairRegsIo <= 2 * kPairRegsLaunch, "register split exceeds the launch");

template <int D, bool BF16, bool VARLEN, bool PAIR = false>
__global__ void __launch_bounds__(kFwdThreads, PAIR ? 2 : 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const FwdArgs args) {
    using C = FwdCfg<D, PAIR>;
    constexpr int NB = C::kSBuf;
    // Sleep between an issuing thread's barrier polls.  The paired form's tiles form
    // one serial S -> softmax -> PV chain per CTA, so its issuers poll without
    // sleeping (try_wait itself suspends the thread for a while): a wake-up
    // that waited out a sleep lengthened every link of the chain (+3-5 % on paired
    // grids without it; neutral on the one-CTA form, which keeps the sleep).
    constexpr uint32_t kIssuerSleepNs = PAIR ? 0u : 32u;
    using PK = Pack<BF16>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sb = raw + pad;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Launch order (the hardware hands out CTAs in linear block order): consecutive
    // CTAs take consecutive row blocks of one head, heaviest causal block first, so the
    // CTAs resident at any time share a few heads' K/V in L2.  With head_group > 1 (a
    // grid of a few waves) the (row block, head) pairs are walked head_group heads at a
    // time instead, and within a group row block by row block across the group's heads,
    // so that the heaviest blocks of the last heads do not start at the end of the launch.
    int bx = (int)blockIdx.x, by = (int)blockIdx.y;
    if (args.head_group > 1) {
        const int per = (int)gridDim.x, g = args.head_group;
        const int lin = (int)blockIdx.y * per + (int)blockIdx.x;
        const int chunk = lin / (g * per), rem = lin - chunk * g * per;
        const int gh = min(g, (int)gridDim.y - chunk * g);  // heads in this group
        bx = rem / gh;
        by = chunk * g + rem % gh;
    }
    int bh = by;
    const int causal = args.causal;
    int q0, Nq, Nk, kvh;
    int q_tok = 0, k_tok = 0;  // VARLEN: first token of this sequence in q and in k, v
    if constexpr (VARLEN) {
        int seq, blk = -1;
        if (args.work != nullptr) {
            // Planned grid: bx indexes the work list, by is the head.
            if (bx >= args.work[0]) return;  // past the list (the whole CTA)
            const int2 w = reinterpret_cast<const int2 *>(args.work + 2)[bx];
            seq = w.x;
            blk = w.y;
            bh = seq * args.H + by;
        } else {
            seq = bh / args.H;
        }
        q_tok = args.cu_q[seq];
        k_tok = args.cu_k[seq];
        Nq = args.cu_q[seq + 1] - q_tok;
        Nk = args.cu_k[seq + 1] - k_tok;
        const int num_m = (Nq + kFwdBr - 1) / kFwdBr;
        // Unplanned grid: row blocks past this sequence's own ones hold no row (q0 >= Nq).
        if (blk < 0) blk = bx < num_m ? num_m - 1 - bx : -1;
        q0 = blk >= 0 ? blk * kFwdBr : max(Nq, 0);
        kvh = (bh % args.H) / args.group;  // K/V head index within the token's heads
    } else {
        q0 = (args.num_m - 1 - bx) * kFwdBr;
        Nq = args.Nq;
        Nk = args.Nk;
        kvh = kv_head(bh, args.H, args.group);  // the K/V head this query head reads
    }
    // A variable-length grid is sized by the longest sequence: a CTA past its own
    // sequence's row blocks holds no row and leaves before touching shared or tensor
    // memory (the whole CTA takes this branch together).
    if (VARLEN && q0 >= Nq) return;
    const int n = fwd_tile_count(q0, Nq, Nk, causal);
    const int jm = fwd_first_masked_tile(q0, Nq, Nk, causal);

    auto bar = [&](int idx) -> uint32_t { return sb + C::kOffBar + 8u * (uint32_t)idx; };
    constexpr int S_ = C::kStages;
    constexpr int B_QFULL = 0;
    auto B_KFULL = [](int s) { return 1 + s; };
    auto B_KEMPTY = [](int s) { return 1 + S_ + s; };
    auto B_VFULL = [](int s) { return 1 + 2 * S_ + s; };
    auto B_VEMPTY = [](int s) { return 1 + 3 * S_ + s; };
    auto B_SFULL = [](int b) { return 1 + 4 * S_ + b; };   // S(t) in S[b], b = t % 3
    auto B_PFULL = [](int b) { return 4 + 4 * S_ + b; };   // P(j) in S[b] (one arrival per softmax warp)
    auto B_PVDONE = [](int b) { return 7 + 4 * S_ + b; };  // PV(j) complete, b = j % 3
    constexpr int B_OFINAL = 10 + 4 * S_;                  // last PV complete
    auto B_MMAFIN = [](int w) { return 11 + 4 * S_ + w; }; // every MMA of issuer w complete
    volatile uint32_t *tmem_holder = reinterpret_cast<volatile uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
    int *status = args.status;

    // The producer's lane initialises the barriers and, before the CTA-wide sync that
    // waits for the tensor-memory allocation, already sends out the Q tile and the
    // first K tiles (their slots are fresh, so no empty-slot wait is needed): their
    // latency overlaps the allocation and the sync.  No other thread touches a
    // barrier before that sync.
    constexpr int kProducer = kWarpTma * 32;
    const int n_first = min(n, C::kAhead);  // K tiles loaded before the sync
    if (threadIdx.x == kProducer) {
        mbar_init(bar(B_QFULL), 1);
        for (int s = 0; s < S_; ++s) {
            mbar_init(bar(B_KFULL(s)), 1);
            mbar_init(bar(B_KEMPTY(s)), 1);
            mbar_init(bar(B_VFULL(s)), 1);
            mbar_init(bar(B_VEMPTY(s)), 1);
        }
        for (int b = 0; b < 3; ++b) {
            mbar_init(bar(B_SFULL(b)), 1);
            mbar_init(bar(B_PFULL(b)), 4);
            mbar_init(bar(B_PVDONE(b)), 1);
        }
        mbar_init(bar(B_OFINAL), 1);
        mbar_init(bar(B_MMAFIN(0)), 1);
        mbar_init(bar(B_MMAFIN(1)), 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmO);
        if (n > 0) {
            mbar_arrive_expect_tx(bar(B_QFULL), C::kQBytes);
            for (int b = 0; b < C::kBlocks; ++b)
                if constexpr (VARLEN)
                    tma_load_3d(sb + C::kOffQ + b * C::kQBlockBytes, &tmQ, b * 64, bh % args.H, q_tok + q0, bar(B_QFULL));
                else
                    tma_load_3d(sb + C::kOffQ + b * C::kQBlockBytes, &tmQ, b * 64, q0, bh, bar(B_QFULL));
            for (int t = 0; t < n_first; ++t) {
                mbar_arrive_expect_tx(bar(B_KFULL(t)), C::kTileBytes);
                for (int b = 0; b < C::kBlocks; ++b)
                    if constexpr (VARLEN)
                        tma_load_3d(sb + C::kOffK + t * C::kTileBytes + b * C::kKVBlockBytes, &tmK, b * 64, kvh,
                                    k_tok + t * kFwdBc, bar(B_KFULL(t)));
                    else
                        tma_load_3d(sb + C::kOffK + t * C::kTileBytes + b * C::kKVBlockBytes, &tmK, b * 64,
                                    t * kFwdBc, kvh, bar(B_KFULL(t)));
            }
        }
    }
    if (warp == kWarpPv) {
        tmem_alloc(sb + C::kOffMisc, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    constexpr uint32_t hi = sdesc_hi_sw128(1024);  // 8 rows x 128 B per core group

    auto producer_role = [&]() {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && n > 0) {
            // The Q tile and K_0 .. K_{n_first-1} went out before the sync (first use of each slot).
            uint32_t pend_k = (1u << n_first) - 1u, pend_v = 0;  // slots with a load issued, per ring
            uint32_t par_k = 0, par_v = 0;                        // phase parity of the last load into each slot
            // Tile `tile` of K (V) goes to slot tile % S of its ring, in the order the two
            // MMA streams consume them: K_0 .. K_{A-1}, then V_j, K_{j+A} for j = 0, 1, ...
            // (A = kAhead: 3, or 2 in the paired form).
            auto load = [&](bool is_v, int tile) -> bool {
                const int s = tile % S_;
                const uint32_t it = (uint32_t)(tile / S_);
                if (!mbar_wait_backoff(bar(is_v ? B_VEMPTY(s) : B_KEMPTY(s)), (it & 1u) ^ 1u, abort_flag, status, 64))
                    return false;
                const uint32_t full = bar(is_v ? B_VFULL(s) : B_KFULL(s));
                mbar_arrive_expect_tx(full, C::kTileBytes);
                const uint32_t dst = sb + (is_v ? C::kOffV : C::kOffK) + s * C::kTileBytes;
                for (int b = 0; b < C::kBlocks; ++b)
                    if constexpr (VARLEN)
                        tma_load_3d(dst + b * C::kKVBlockBytes, is_v ? &tmV : &tmK, b * 64, kvh, k_tok + tile * kFwdBc, full);
                    else
                        tma_load_3d(dst + b * C::kKVBlockBytes, is_v ? &tmV : &tmK, b * 64, tile * kFwdBc, kvh, full);
                (is_v ? pend_v : pend_k) |= 1u << s;
                uint32_t &par = is_v ? par_v : par_k;
                par = (par & ~(1u << s)) | ((it & 1u) << s);
                return true;
            };
            bool ok = true;
            for (int j = 0; ok && j < n; ++j) ok = load(true, j) && (j + C::kAhead >= n || load(false, j + C::kAhead));
            // Every load issued must land before the CTA may exit.
            volatile int no_abort = 0;
            mbar_wait_bounded(bar(B_QFULL), 0, &no_abort, status);
            for (int s = 0; s < S_; ++s) {
                if (pend_k & (1u << s)) mbar_wait_bounded(bar(B_KFULL(s)), (par_k >> s) & 1u, &no_abort, status);
                if (pend_v & (1u << s)) mbar_wait_bounded(bar(B_VFULL(s)), (par_v >> s) & 1u, &no_abort, status);
            }
        }
    };
    auto s_issuer_role = [&]() {
        // ------------------------------------------------------------ MMA issuer: S stream
        if (lane == 0 && n > 0) {
            constexpr uint32_t idesc_qk = idesc_f16(128, kFwdBc, BF16, false);
            const uint32_t q_lo = sdesc_lo(sb + C::kOffQ, 16);  // K-major: LBO unused
            const uint32_t k_lo = sdesc_lo(sb + C::kOffK, 16);
            bool ok = mbar_wait_bounded(bar(B_QFULL), 0, abort_flag, status);
            for (int t = 0; ok && t < n; ++t) {
                const int b = t % NB, s = t % S_;
                // S[b] is free once PV(t-NB) has read P(t-NB) from it.
                if (t >= NB) ok = mbar_wait_backoff(bar(B_PVDONE(b)), (uint32_t)(t / NB - 1) & 1u, abort_flag, status, 2 * kIssuerSleepNs);
                ok = ok && mbar_wait_backoff(bar(B_KFULL(s)), (uint32_t)(t / S_) & 1u, abort_flag, status, 2 * kIssuerSleepNs);
                if (!ok) break;
                tc_fence_after();
                // S(t) = Q K_t^T: K-major A and B, 16 of the d columns per instruction.
                const uint32_t kt_lo = k_lo + (uint32_t)(s * (C::kTileBytes >> 4));
                const uint32_t d_s = tmem + C::tmem_s(b);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off_q = ((k >> 2) * C::kQBlockBytes + (k & 3) * 32) >> 4;
                    const uint32_t off_k = ((k >> 2) * C::kKVBlockBytes + (k & 3) * 32) >> 4;
                    umma_ss_w(d_s, q_lo + off_q, hi, kt_lo + off_k, hi, idesc_qk, k > 0 ? 1u : 0u);
                }
                umma_commit(bar(B_SFULL(b)));
                umma_commit(bar(B_KEMPTY(s)));
            }
            // Tensor memory may be freed only after every issued MMA completed.
            umma_commit(bar(B_MMAFIN(1)));
            volatile int no_abort = 0;
            mbar_wait_bounded(bar(B_MMAFIN(1)), 0, &no_abort, status);
        }
    };
    auto pv_issuer_role = [&]() {
        // ------------------------------------------------------------ MMA issuer: PV stream
        if (lane == 0 && n > 0) {
            constexpr uint32_t idesc_pv = idesc_f16(128, D, BF16, true);
            const uint32_t v_lo = sdesc_lo(sb + C::kOffV, C::kKVBlockBytes);  // MN-major: LBO = 64-col block
            const uint32_t d_o = tmem + C::kTmemO;
            bool ok = true;
            for (int j = 0; ok && j < n; ++j) {
                const int b = j % NB, s = j % S_;
                ok = mbar_wait_backoff(bar(B_PFULL(b)), (uint32_t)(j / NB) & 1u, abort_flag, status, kIssuerSleepNs) &&
                     mbar_wait_backoff(bar(B_VFULL(s)), (uint32_t)(j / S_) & 1u, abort_flag, status, kIssuerSleepNs);
                if (!ok) break;
                tc_fence_after();
                // O += P(j) V_j: P from S[b] (the remainder too on masked tiles), V as an
                // MN-major operand, 16 keys per instruction.
                const uint32_t vt_lo = v_lo + (uint32_t)(s * (C::kTileBytes >> 4));
                const uint32_t p_t = tmem + C::tmem_s(b);
#pragma unroll
                for (int k = 0; k < kFwdBc / 16; ++k)
                    umma_ts_w(d_o, p_t + 8 * k, vt_lo + ((k * 2048) >> 4), hi, idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
                if (j >= jm) {
#pragma unroll
                    for (int k = 0; k < kFwdBc / 16; ++k)
                        umma_ts_w(d_o, p_t + 64 + 8 * k, vt_lo + ((k * 2048) >> 4), hi, idesc_pv, 1u);
                }
                umma_commit(bar(B_PVDONE(b)));
                umma_commit(bar(B_VEMPTY(s)));
            }
            if (ok) umma_commit(bar(B_OFINAL));
            umma_commit(bar(B_MMAFIN(0)));
            volatile int no_abort = 0;
            mbar_wait_bounded(bar(B_MMAFIN(0)), 0, &no_abort, status);
        }
    };
    auto softmax_role = [&]() {
        // ------------------------------------------------------------ softmax / correction / epilogue
        const int quarter = warp;  // TMEM lanes [32*quarter, 32*quarter+32) belong to this warp
        const int i = q0 + quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t o_addr = lane_base + C::kTmemO;
        const int lim = causal ? min(i + (Nk - Nq), Nk - 1) : Nk - 1;  // last key row i may see
        const float sl2 = args.scale_log2;
        float m = -INFINITY;  // running (possibly stale) max of scale*log2(e)*s
        float l = 0.f;        // running sum of 2^(scale*log2(e)*s - m)
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            const int b = j % NB;
            ok = __all_sync(0xffffffffu,
                            mbar_wait_bounded(bar(B_SFULL(b)), (uint32_t)(j / NB) & 1u, abort_flag, status));
            if (!ok) break;
            tc_fence_after();
            const uint32_t s_addr = lane_base + C::tmem_s(b);
            // Two instances of the same step, so the unmasked (common) tile carries no
            // predicated mask or remainder instructions.
            const RowStep r = j >= jm ? softmax_tile_masked<BF16>(s_addr, j * kFwdBc, lim, sl2, m, l)
                                      : softmax_tile<false, BF16>(s_addr, 0, 0, sl2, m, l);
            m = r.m;
            l = r.l;
            if (r.rescale && j > 0) {
                // O must hold PV(0..j-1) in full before it is scaled.
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(B_PVDONE((j - 1) % NB)), (uint32_t)((j - 1) / NB) & 1u,
                                                               abort_flag, status));
                if (!ok) break;
                tc_fence_after();
                rescale_o<D>(o_addr, r.alpha);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_PFULL(b)));
        }
        if (ok && n > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(B_OFINAL), 0, abort_flag, status));
            tc_fence_after();
        }
        // Epilogue: O = O~ / l (0 for a row that saw no key), LSE = m ln2 + ln l.  The
        // rows go through shared memory (K ring slot 0: every S MMA, hence every read
        // of the K ring, completed before the last PV did) in the layout of a Q or K
        // tile, and leave as TMA stores of whole 128-byte rows; rows past Nq are clipped
        // by the tensor map.  A packed batch's last row block of a sequence stops short
        // of the tile (its box would run into the next sequence's rows): its rows are
        // stored directly.
        const bool staged = !VARLEN || q0 + kFwdBr <= Nq;
        const bool valid = i < Nq;
        const int row = quarter * 32 + lane;
        const bool work = ok && __any_sync(0xffffffffu, valid);  // the same on the whole warp
        const float inv = (l > 0.f) ? 1.f / l : 0.f;
        const size_t orow = VARLEN ? (size_t)(q_tok + i) * args.H + bh % args.H : (size_t)bh * Nq + i;
        typename PK::T *orow_g = reinterpret_cast<typename PK::T *>(args.o) + orow * D;
        uint8_t *stage_row = smem + C::kOffK + row * 128;
        // One 64-column block at a time: once every softmax warp has staged block b,
        // its TMA store goes out and reads shared memory while the next block is packed.
#pragma unroll 1
        for (int b = 0; b < C::kBlocks; ++b) {
            if (work) {
#pragma unroll 1
                for (int c = 2 * b; c < 2 * b + 2; ++c) {
                    uint32_t ov[32];
                    if (n > 0) {
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
                    if (staged) {
                        // columns [32c, 32c+32): 64-column block b, 16-byte chunks 4(c%2)..4(c%2)+3,
                        // chunk k of row r at r*128 + 16*(k ^ (r mod 8)) (the 128-byte swizzle)
                        uint8_t *blk = stage_row + b * C::kKVBlockBytes;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int k = 4 * (c & 1) + e;
                            *reinterpret_cast<uint4 *>(blk + 16 * (k ^ (row & 7))) =
                                make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                        }
                    } else if (valid) {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow_g + 32 * c);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                    }
                }
            }
            if (staged) {
                // Every softmax warp arrives (whatever its rows or its wait outcomes), so the
                // barrier always completes; the stores go out only if no warp gave up a wait.
                fence_proxy_async_smem();
                const bool all_ok = named_bar_and(1, 128, ok);
                if (all_ok && threadIdx.x == 0) {
                    if constexpr (VARLEN)
                        tma_store_3d(&tmO, sb + C::kOffK + b * C::kKVBlockBytes, b * 64, bh % args.H, q_tok + q0);
                    else
                        tma_store_3d(&tmO, sb + C::kOffK + b * C::kKVBlockBytes, b * 64, q0, bh);
                    bulk_commit();
                }
            }
        }
        if (work && valid && args.lse != nullptr) {
            const float m_fin = (m == -INFINITY) ? 0.f : m;
            const size_t lrow = VARLEN ? (size_t)(bh % args.H) * args.total_q + q_tok + i : (size_t)bh * Nq + i;
            args.lse[lrow] = (l > 0.f) ? m_fin * 0.69314718055994531f + logf(l) : -INFINITY;
        }
        // The stores must have read shared memory before the CTA may exit.
        if (staged && threadIdx.x == 0) bulk_wait_read();
    };
    // The roles.  Paired form: the producer/issuer warpgroup (warps 4-7) gives
    // registers to the softmax warpgroup before either splits into its roles.
    if constexpr (PAIR) {
        if (warp >= 4) {
            regs_decrease<kPairRegsIo>();
            if (warp == kWarpTma) producer_role();
            else if (warp == kWarpS) s_issuer_role();
            else if (warp == kWarpPv) pv_issuer_role();
        } else {
            regs_increase<kPairRegsSoftmax>();
            softmax_role();
        }
    } else {
        if (warp == kWarpTma) producer_role();
        else if (warp == kWarpS) s_issuer_role();
        else if (warp == kWarpPv) pv_issuer_role();
        else if (warp < 4) softmax_role();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpPv) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool BF16, bool VARLEN, bool PAIR = false>
static cudaError_t launch_fwd_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                                const CUtensorMap &to, const FwdArgs &a, int num_m, int rows_y, cudaStream_t stream) {
    using C = FwdCfg<D, PAIR>;
    auto kern = fa_fwd_kernel<D, BF16, VARLEN, PAIR>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (PAIR) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
    }
    dim3 grid((unsigned)num_m, (unsigned)rows_y, 1);
    return launch_kernel(kern, grid, dim3(kFwdThreads), C::kSmemBytes, stream, tq, tk, tv, to, a);
}

template <bool VARLEN>
static cudaError_t launch_fwd_any(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk,
                                  const CUtensorMap &tv, const CUtensorMap &to, const FwdArgs &a, int rows_y,
                                  cudaStream_t stream, bool pair = false) {
    if (d == 64 && pair && !VARLEN)
        return bf16 ? launch_fwd_t<64, true, false, true>(tq, tk, tv, to, a, a.num_m, rows_y, stream)
                    : launch_fwd_t<64, false, false, true>(tq, tk, tv, to, a, a.num_m, rows_y, stream);
    if (d == 64) return bf16 ? launch_fwd_t<64, true, VARLEN>(tq, tk, tv, to, a, a.num_m, rows_y, stream)
                             : launch_fwd_t<64, false, VARLEN>(tq, tk, tv, to, a, a.num_m, rows_y, stream);
    return bf16 ? launch_fwd_t<128, true, VARLEN>(tq, tk, tv, to, a, a.num_m, rows_y, stream)
                : launch_fwd_t<128, false, VARLEN>(tq, tk, tv, to, a, a.num_m, rows_y, stream);
}

cudaError_t launch_fwd(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &to, const FwdArgs &a, int BH, cudaStream_t stream, bool pair) {
    return launch_fwd_any<false>(d, bf16, tq, tk, tv, to, a, BH, stream, pair);
}

cudaError_t launch_fwd_varlen(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                              const CUtensorMap &to, const FwdArgs &a, int num_seqs, cudaStream_t stream) {
    return launch_fwd_any<true>(d, bf16, tq, tk, tv, to, a, num_seqs * a.H, stream);
}

// Work list of a variable-length batch (one CTA of 1024 threads).  Sequence s has
// nb_s = ceil(len(s) / 128) blocks of 128 tokens; the sequences are ordered by nb_s
// descending (ties by index) and each sequence's blocks last-first (the forward's
// heaviest causal row block is its last) or first-first (the backward's heaviest
// causal key block is its first), so that the longest work starts first.  Each
// thread finds its sequences' place in that order with one pass over all the block
// counts (num_seqs^2 / 1024 steps per thread).
__global__ void __launch_bounds__(1024) fa_varlen_plan_kernel(const int *cu, int num_seqs, int *work, int last_first) {
    int2 *list = reinterpret_cast<int2 *>(work + 2);
    int total = 0;
    for (int s = threadIdx.x; s < num_seqs; s += blockDim.x) {
        const int nb = (cu[s + 1] - cu[s] + kFwdBr - 1) / kFwdBr;
        int start = 0;
        for (int t = 0; t < num_seqs; ++t) {
            const int nt = (cu[t + 1] - cu[t] + kFwdBr - 1) / kFwdBr;
            if (nt > nb || (nt == nb && t < s)) start += nt;
        }
        for (int b = 0; b < nb; ++b) list[start + b] = make_int2(s, last_first ? nb - 1 - b : b);
        total += nb;
    }
    // the list's length: the sum of every thread's block counts
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    __shared__ int warp_total[32];
    if ((threadIdx.x & 31) == 0) warp_total[threadIdx.x >> 5] = total;
    __syncthreads();
    if (threadIdx.x == 0) {
        int sum = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) sum += warp_total[w];
        work[0] = sum;
    }
}

cudaError_t launch_varlen_plan(const int *cu, int num_seqs, int *work, bool last_first, cudaStream_t stream) {
    return launch_kernel(fa_varlen_plan_kernel, dim3(1), dim3(1024), 0, stream, cu, num_seqs, work, last_first ? 1 : 0);
}

cudaError_t launch_fwd_varlen_planned(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk,
                                     const CUtensorMap &tv, const CUtensorMap &to, const FwdArgs &a, int *work,
                                     int capacity, cudaStream_t stream) {
    cudaError_t e = launch_varlen_plan(a.cu_q, a.num_seqs, work, true, stream);
    if (e != cudaSuccess) return e;
    FwdArgs b = a;
    b.work = work;
    b.num_m = capacity;
    return launch_fwd_any<true>(d, bf16, tq, tk, tv, to, b, a.H, stream);
}

}  // namespace fa
