// fa_fwd_sm103.cu -- fused exact attention forward on sm_103a tensor cores.
//
// One CTA computes one 128-row Q tile of one (batch, head):
//   O_i = sum_j softmax_j(scale * q_i . k_j + mask) v_j,  LSE_i = m_i + ln l_i
// following the FlashAttention-2 forward ("6.2 FlashAttention V2 explained",
// §6): the Q tile stays on chip, K/V tiles stream past it, a running row max m
// and row sum l are kept per row, the accumulator is rescaled by
// exp(m_old - m_new) and divided by l once at the end (§3.2; "02 · FA2", §1).
// Causal masking visits only K/V tiles up to the diagonal and masks element-wise
// only on tiles that straddle it or the ragged Nk tail (§5.3; "02 · FA2", §4).
//
// Roles (warp specialisation, 6 warps):
//   warp 0     TMA producer: Q once, then K_0, V_0, K_1, V_1, ... through a
//              ring of shared-memory slots guarded by full/empty mbarriers.
//   warp 1     owns tensor memory; one lane issues tcgen05.mma:
//              S_j = Q K_j^T into one of two TMEM S buffers (fp32), and
//              O += P_j V_j with P read from TMEM (the A operand) and V from
//              shared memory (MN-major B operand).
//   warps 2-5  softmax, one thread per query row (TMEM lane = row): load the
//              S row, mask, update (m, l) in base 2, write P as 16-bit into
//              TMEM, rescale the O row by alpha when the max moved, and in the
//              epilogue normalise by 1/l and write O and LSE.
// The MMA of S_{j+1} runs while the softmax of tile j runs (two S buffers).
//
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O [256,256+d),
// P [384,448) and, on masked tiles, P_lo [448,512).  On a masked tile P is
// written as a 16-bit head plus a 16-bit remainder (P = P_hi + P_lo) and both
// are multiplied into O: rows with few visible keys are then not limited by
// the 16-bit rounding of their few large weights.
//
// Every mbarrier wait is bounded (%globaltimer); on expiry the CTA records
// the timeout in the status word, stops issuing work, waits (bounded) for its
// in-flight TMA loads and MMAs, frees tensor memory and exits.
#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {

constexpr int kFwdThreads = 192;

template <int D>
struct FwdCfg {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int kStages = (D == 128) ? 4 : 6;
    static constexpr int kBlocks = D / 64;               // 128-byte swizzle blocks per row
    static constexpr int kQBlockBytes = kFwdBr * 128;    // one 64-column block of the Q tile
    static constexpr int kKVBlockBytes = kFwdBc * 128;   // one 64-column block of a K/V tile
    static constexpr int kQBytes = kFwdBr * D * 2;
    static constexpr int kTileBytes = kFwdBc * D * 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffRing = kQBytes;
    static constexpr int kOffBar = kOffRing + kStages * kTileBytes;
    // barriers: q_full, full[S], empty[S], s_full[2], p_full[2], o_done, mma_fin
    static constexpr int kNumBars = 1 + 2 * kStages + 2 + 2 + 1 + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    // Unused tail after the last slot: keeps any tensor-core operand read that a
    // descriptor could reach from the last slot inside this CTA's allocation.
    static constexpr int kGuardBytes = 32768;
    static constexpr int kSmemBytes = kOffMisc + 16 + kGuardBytes + 1024;  // + slack to align the base
    static constexpr uint32_t kTmemS0 = 0, kTmemS1 = 128, kTmemO = 256, kTmemP = 384, kTmemPlo = 448;
    static constexpr uint32_t kTmemCols = 512;
};

// Tile j needs element masks when it crosses the ragged end of K or, under
// causal masking, holds a key beyond the first row's last visible key.
__device__ __forceinline__ bool fwd_tile_needs_mask(int j, int q0, int Nq, int Nk, int causal) {
    const int last_key = (j + 1) * kFwdBc - 1;
    return (last_key >= Nk) || (causal && last_key > q0 + (Nk - Nq));
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
    const int bh = blockIdx.x;
    const int m_block = args.num_m - 1 - (int)blockIdx.y;  // heaviest causal tiles first
    const int q0 = m_block * kFwdBr;
    const int Nq = args.Nq, Nk = args.Nk, causal = args.causal;

    int kv_end = Nk;
    if (causal) kv_end = min(Nk, min(q0 + kFwdBr, Nq) + (Nk - Nq));
    const int n_tiles = kv_end > 0 ? (kv_end + kFwdBc - 1) / kFwdBc : 0;

    auto bar = [&](int idx) -> uint32_t { return sb + C::kOffBar + 8u * (uint32_t)idx; };
    const int B_QFULL = 0;
    auto B_FULL = [](int s) { return 1 + s; };
    auto B_EMPTY = [](int s) { return 1 + C::kStages + s; };
    auto B_SFULL = [](int b) { return 1 + 2 * C::kStages + b; };
    auto B_PFULL = [](int b) { return 3 + 2 * C::kStages + b; };
    const int B_ODONE = 5 + 2 * C::kStages;
    const int B_MMAFIN = 6 + 2 * C::kStages;
    volatile uint32_t *tmem_holder = reinterpret_cast<volatile uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
    int *status = args.status;

    if (threadIdx.x == 0) {
        mbar_init(bar(B_QFULL), 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar(B_FULL(s)), 1);
            mbar_init(bar(B_EMPTY(s)), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_SFULL(b)), 1);
            mbar_init(bar(B_PFULL(b)), 128);
        }
        mbar_init(bar(B_ODONE), 1);
        mbar_init(bar(B_MMAFIN), 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(sb + C::kOffMisc, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && n_tiles > 0) {
            uint32_t pend_mask = 0, pend_par = 0;
            mbar_arrive_expect_tx(bar(B_QFULL), C::kQBytes);
            for (int b = 0; b < C::kBlocks; ++b)
                tma_load_3d(sb + C::kOffQ + b * C::kQBlockBytes, &tmQ, b * 64, q0, bh, bar(B_QFULL));
            for (int t = 0; t < 2 * n_tiles; ++t) {
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
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n_tiles > 0) {
            constexpr uint32_t idesc_qk = idesc_f16(128, kFwdBc, BF16, false);
            constexpr uint32_t idesc_pv = idesc_f16(128, D, BF16, true);
            const uint32_t qa = sb + C::kOffQ;
            bool ok = mbar_wait_bounded(bar(B_QFULL), 0, abort_flag, status);
            for (int j = 0; ok && j <= n_tiles; ++j) {
                if (j < n_tiles) {
                    // S_j = Q K_j^T  (K-major A and B, 16 keys of d per instruction)
                    const int t = 2 * j;
                    const int s = t % C::kStages;
                    if (!mbar_wait_bounded(bar(B_FULL(s)), (uint32_t)(t / C::kStages) & 1u, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t ka = sb + C::kOffRing + s * C::kTileBytes;
                    const uint32_t dS = tmem + ((j & 1) ? C::kTmemS1 : C::kTmemS0);
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t off_q = (k >> 2) * C::kQBlockBytes + (k & 3) * 32;
                        const uint32_t off_k = (k >> 2) * C::kKVBlockBytes + (k & 3) * 32;
                        umma_ss(dS, sdesc_sw128(qa + off_q, 16, 1024), sdesc_sw128(ka + off_k, 16, 1024), idesc_qk,
                                k > 0 ? 1u : 0u);
                    }
                    umma_commit(bar(B_SFULL(j & 1)));
                    umma_commit(bar(B_EMPTY(s)));
                }
                if (j > 0) {
                    // O += P_{j-1} V_{j-1}  (P from TMEM, V MN-major from shared memory)
                    const int jj = j - 1;
                    const int t = 2 * jj + 1;
                    const int s = t % C::kStages;
                    if (!mbar_wait_bounded(bar(B_PFULL(jj & 1)), (uint32_t)(jj >> 1) & 1u, abort_flag, status) ||
                        !mbar_wait_bounded(bar(B_FULL(s)), (uint32_t)(t / C::kStages) & 1u, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t va = sb + C::kOffRing + s * C::kTileBytes;
#pragma unroll
                    for (int k = 0; k < kFwdBc / 16; ++k)
                        umma_ts(tmem + C::kTmemO, tmem + C::kTmemP + 8 * k,
                                sdesc_sw128(va + k * 2048, C::kKVBlockBytes, 1024), idesc_pv,
                                (jj > 0 || k > 0) ? 1u : 0u);
                    if (fwd_tile_needs_mask(jj, q0, Nq, Nk, causal)) {
#pragma unroll
                        for (int k = 0; k < kFwdBc / 16; ++k)
                            umma_ts(tmem + C::kTmemO, tmem + C::kTmemPlo + 8 * k,
                                    sdesc_sw128(va + k * 2048, C::kKVBlockBytes, 1024), idesc_pv, 1u);
                    }
                    umma_commit(bar(B_ODONE));
                    umma_commit(bar(B_EMPTY(s)));
                }
            }
            // Tensor memory may be freed only after every issued MMA completed.
            umma_commit(bar(B_MMAFIN));
            volatile int no_abort = 0;
            mbar_wait_bounded(bar(B_MMAFIN), 0, &no_abort, status);
        }
    } else {
        // ------------------------------------------------------------ softmax / correction / epilogue
        const int quarter = warp & 3;  // TMEM lanes [32*quarter, 32*quarter+32) belong to this warp
        const int r = quarter * 32 + lane;
        const int i = q0 + r;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const int lim = causal ? min(i + (Nk - Nq), Nk - 1) : Nk - 1;  // last key row i may see
        const float sl2 = args.scale_log2;
        float m = -INFINITY;  // running max of scale*log2(e)*s
        float l = 0.f;        // running sum of 2^(.. - m)
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            ok = mbar_wait_bounded(bar(B_SFULL(j & 1)), (uint32_t)(j >> 1) & 1u, abort_flag, status);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t sbuf = lane_base + ((j & 1) ? C::kTmemS1 : C::kTmemS0);
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(sbuf + 32 * c, sr[c]);
            tmem_wait_ld();
            const bool masked = fwd_tile_needs_mask(j, q0, Nq, Nk, causal);
            if (masked) {
                const int c0 = j * kFwdBc;
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c0 + c > lim) sr[c >> 5][c & 31] = __float_as_uint(-INFINITY);
            }
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 128; ++c) mx = fmaxf(mx, __uint_as_float(sr[c >> 5][c & 31]));
            const float m_new = fmaxf(m, mx * sl2);
            const float m_d = (m_new == -INFINITY) ? 0.f : m_new;  // never subtract -inf from -inf
            const float alpha = ex2_approx(m - m_d);
            float rs = 0.f;
            uint32_t ph[2][32], pl[2][32];
#pragma unroll
            for (int c = 0; c < 128; c += 2) {
                const float p0 = ex2_approx(fmaf(__uint_as_float(sr[c >> 5][c & 31]), sl2, -m_d));
                const float p1 = ex2_approx(fmaf(__uint_as_float(sr[c >> 5][(c + 1) & 31]), sl2, -m_d));
                rs += p0 + p1;
                const uint32_t h = PK::pack(p0, p1);
                ph[c >> 6][(c >> 1) & 31] = h;
                if (masked) {
                    const float2 hf = PK::unpack(h);
                    pl[c >> 6][(c >> 1) & 31] = PK::pack(p0 - hf.x, p1 - hf.y);
                }
            }
            l = l * alpha + rs;
            m = m_new;
            if (j > 0) {
                // P and O are free once the previous O += P V has completed.
                ok = mbar_wait_bounded(bar(B_ODONE), (uint32_t)(j - 1) & 1u, abort_flag, status);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            tmem_st_32x32b_x32(lane_base + C::kTmemP, ph[0]);
            tmem_st_32x32b_x32(lane_base + C::kTmemP + 32, ph[1]);
            if (masked) {
                tmem_st_32x32b_x32(lane_base + C::kTmemPlo, pl[0]);
                tmem_st_32x32b_x32(lane_base + C::kTmemPlo + 32, pl[1]);
            }
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t orow[32];
                    tmem_ld_32x32b_x32(lane_base + C::kTmemO + 32 * c, orow);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) orow[e] = __float_as_uint(__uint_as_float(orow[e]) * alpha);
                    tmem_st_32x32b_x32(lane_base + C::kTmemO + 32 * c, orow);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(B_PFULL(j & 1)));
        }
        if (ok && n_tiles > 0) {
            ok = mbar_wait_bounded(bar(B_ODONE), (uint32_t)(n_tiles - 1) & 1u, abort_flag, status);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
        }
        if (ok) {
            // Epilogue: O = O~ / l (0 for a row that saw no key), LSE = m ln2 + ln l.
            const bool valid = i < Nq;
            const float inv = (l > 0.f) ? 1.f / l : 0.f;
            typename PK::T *orow_g = reinterpret_cast<typename PK::T *>(args.o) + ((size_t)bh * Nq + i) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t ov[32];
                if (n_tiles > 0) {
                    tmem_ld_32x32b_x32(lane_base + C::kTmemO + 32 * c, ov);
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
                const float m_d = (m == -INFINITY) ? 0.f : m;
                args.lse[(size_t)bh * Nq + i] = (l > 0.f) ? m_d * 0.69314718055994531f + logf(l) : -INFINITY;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
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
    dim3 grid((unsigned)BH, (unsigned)a.num_m, 1);
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
