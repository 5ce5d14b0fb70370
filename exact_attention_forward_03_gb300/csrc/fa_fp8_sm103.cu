// fa_fp8_sm103.cu -- FP8 (E4M3) attention forward on sm_103a tensor cores, and
// the block quantization that feeds it.
//
// The pages run both products of the forward in FP8 (E4M3) and keep per-block
// scale factors so that small values do not vanish ("Flash Attention (4)"
// §5.4; the FP8-underflow exercise of §8.3).  Here:
//
//   quantization (fa_fp8_quant_kernel): for every block of 128 rows of one head,
//     s = amax / 448 (fp32; 1 for an all-zero block) and code = E4M3(x / s),
//     round to nearest even, saturating at 448.  Q and K keep the [BH, N, d]
//     layout; V is written transposed, [BH, d, N_pad] with N_pad a multiple of
//     128, so that it is a K-major operand of P V like K is of Q K^T.
//
//   attention (fa_fwd_fp8_kernel), the structure of the 16-bit forward
//   (fa_fwd_sm103.cu): one 128-row Q tile per CTA, K/V tiles streamed by TMA,
//   three score buffers in tensor memory, separate S and PV issuing threads:
//     S(j)  = Q8 K8_j^T on tcgen05 kind::f8f6f4 (fp32 accumulate), so the true
//             scores are scale * s_q * s_k(j) * S(j): that factor (and log2 e)
//             is applied per tile in fp32 by the softmax;
//     P(j)  = 2^(score log2 e - m) against a running max m taken exactly on
//             every tile (O is rescaled when a row max grows by more than a
//             factor 2, so every p <= 2);
//     O    += E4M3(P(j) * kappa_j) V8_j, kappa_j = 2^7 * s_v(j) / max_j s_v(j),
//             which folds V's per-block scale into P and keeps P * kappa <= 256
//             inside the format; l sums the unrounded fp32 P;
//     O     = O * (max_j s_v(j) / 2^7) / l,  LSE = m ln 2 + ln l.
//   Head dimension 128 only: a Q, K or V^T tile row is then exactly one 128-byte
//   swizzle row.
#include <algorithm>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {

constexpr int kFp8Threads = 256;
constexpr int kFp8WarpTma = 4, kFp8WarpPv = 5, kFp8WarpS = 6;
constexpr float kFp8RescaleThreshold = 1.0f;  // log2 units: p <= 2
constexpr float kFp8PScale = 128.0f;           // 2^7
constexpr int kFp8Stages = 4;

struct Fp8Cfg {
    static constexpr int kTileBytes = 128 * 128;  // 128 rows of 128 one-byte elements
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kTileBytes;
    static constexpr int kOffV = kOffK + kFp8Stages * kTileBytes;
    static constexpr int kOffBar = kOffV + kFp8Stages * kTileBytes;
    static constexpr int kNumBars = 1 + 4 * kFp8Stages + 9 + 1 + 2;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
    __device__ static constexpr uint32_t tmem_s(int b) { return 128u * b; }
    static constexpr uint32_t kTmemO = 384;
    static constexpr uint32_t kTmemCols = 512;
};

// Instruction descriptor for kind::f8f6f4: fp32 D (bits 4-5 = 1), A and B E4M3
// (format 0 in bits 7-9 and 10-12), both K-major, N >> 3 in 17-22, M >> 4 in 24-28.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_ss_f8(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                           uint32_t b_hi, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "mov.b64 da, {%1, %2};\n\t"
        "mov.b64 db, {%3, %4};\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
        "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_ts_f8(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "mov.b64 db, {%2, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], db, %4, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Four fp32 values to E4M3 codes (round to nearest even, saturating), byte k of
// the result holding value k.
__device__ __forceinline__ uint32_t pack_e4m3x4(float v0, float v1, float v2, float v3) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(v1), "f"(v0));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(v3), "f"(v2));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

// ----------------------------------------------------------------------------- quantization
// x / s rounded to the nearest fp32, given y = 1/s rounded to the nearest fp32:
// two residual corrections with exact FMA residuals.  q0 = x y is within 1.5 ulp
// of x / s, q1 = q0 + (x - s q0) y within one ulp, and by Markstein's theorem
// (P. Markstein, "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Develop. 34(1), 1990) q1 + (x - s q1) y rounded is the
// rounded quotient, provided nothing overflows or underflows on the way.  The
// quantizer divides every element of a block by the block's one s, so the
// reciprocal is taken once per block and each element costs one multiply and four
// FMAs.  The sign is taken from x (s > 0): the corrections would turn x = -0 into
// +0, and a quotient that underflows to zero keeps its sign.
__device__ __forceinline__ float div_rn_by(float x, float s, float y) {
    const float q0 = __fmul_rn(x, y);
    const float r0 = __fmaf_rn(-q0, s, x);
    const float q1 = __fmaf_rn(r0, y, q0);
    const float r1 = __fmaf_rn(-q1, s, x);
    return copysignf(__fmaf_rn(r1, y, q1), x);
}

// One CTA per block of 128 rows of one head (blockIdx.x = block, blockIdx.y = head).
// Global memory is only touched with lane-consecutive 16-byte accesses: the
// block's 32 KB come in as 2048 consecutive chunks, go to shared memory with row
// r's chunk j at r * 256 + 16 (j ^ (r mod 16)) (the XOR keeps both the writes and
// the per-row reads below free of bank conflicts), thread t then takes row t / 2,
// columns 64 (t mod 2) ... + 63, and the codes leave through the same buffer:
// row-major with the 16-byte chunk k of row r at r * 128 + 16 (k ^ (r mod 8)), or
// for V transposed, [column][row], one 128-byte output row per head-dim index.
template <bool BF16, bool TRANSPOSE>
__global__ void __launch_bounds__(256, 3) fa_fp8_quant_kernel(const Fp8QuantArgs a) {
    using PK = Pack<BF16>;
    __shared__ float warp_max[8];
    __shared__ __align__(16) uint8_t xs[128 * 256];
    const int t = threadIdx.x;
    const int blk = blockIdx.x, bh = blockIdx.y;
    const int rows = min(128, a.N - blk * 128);  // rows of this block inside the tensor
    const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(a.x) +
                                                       ((size_t)bh * a.N + (size_t)blk * 128) * 256);
    {
        uint4 v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int id = t + 256 * e;  // chunk id: row id / 16, chunk id % 16
            v[e] = (id >> 4) < rows ? src[id] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int id = t + 256 * e, row = id >> 4, j = id & 15;
            *reinterpret_cast<uint4 *>(xs + row * 256 + ((j ^ (row & 15)) << 4)) = v[e];
        }
    }
    __syncthreads();
    const int r = t >> 1, half = t & 1;
    float x[64];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int j = half * 8 + e;
        const uint4 u = *reinterpret_cast<const uint4 *>(xs + r * 256 + ((j ^ (r & 15)) << 4));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = PK::unpack(w[k]);
            x[8 * e + 2 * k] = f.x;
            x[8 * e + 2 * k + 1] = f.y;
        }
    }
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < 64; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((t & 31) == 0) warp_max[t >> 5] = amax;
    __syncthreads();  // also: every thread has read its inputs out of xs
    amax = warp_max[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) amax = fmaxf(amax, warp_max[w]);
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    if (t == 0) a.scales[(size_t)bh * a.num_blocks + blk] = s;
    uint32_t c[16];
    if (s >= 0x1p-60f && s <= 0x1p100f) {
        // With 2^-60 <= s <= 2^100, 1/s and every product stay finite, and for each x
        // whose quotient can round to a nonzero code (|x / s| >= 2^-10) the residuals
        // (about 2^-24 |x| >= 2^-94) stay normal; smaller quotients give a signed
        // zero code whatever their last bits.
        const float y = __frcp_rn(s);
#pragma unroll
        for (int e = 0; e < 16; ++e)
            c[e] = pack_e4m3x4(div_rn_by(x[4 * e], s, y), div_rn_by(x[4 * e + 1], s, y),
                               div_rn_by(x[4 * e + 2], s, y), div_rn_by(x[4 * e + 3], s, y));
    } else {
#pragma unroll
        for (int e = 0; e < 16; ++e)
            c[e] = pack_e4m3x4(__fdiv_rn(x[4 * e], s), __fdiv_rn(x[4 * e + 1], s), __fdiv_rn(x[4 * e + 2], s),
                               __fdiv_rn(x[4 * e + 3], s));
    }
    if constexpr (!TRANSPOSE) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int k = 4 * half + e;  // 16-byte chunk of the 128-byte code row
            *reinterpret_cast<uint4 *>(xs + r * 128 + ((k ^ (r & 7)) << 4)) =
                make_uint4(c[4 * e], c[4 * e + 1], c[4 * e + 2], c[4 * e + 3]);
        }
        __syncthreads();
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(a.x8) + ((size_t)bh * a.N + (size_t)blk * 128) * 128);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int id = t + 256 * e, row = id >> 3, k = id & 7;
            if (row < rows) dst[id] = *reinterpret_cast<const uint4 *>(xs + row * 128 + ((k ^ (row & 7)) << 4));
        }
    } else {
        // [column][row]: rows past N carry x = 0, so code 0 (the padding the
        // transposed layout asks for)
#pragma unroll
        for (int e = 0; e < 64; ++e) xs[(64 * half + e) * 128 + r] = (uint8_t)(c[e >> 2] >> (8 * (e & 3)));
        __syncthreads();
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int id = t + 256 * e, col = id >> 3, k = id & 7;
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(a.x8) + ((size_t)bh * 128 + col) * a.ld_t +
                                                   (size_t)blk * 128 + 16 * k);
            *dst = *reinterpret_cast<const uint4 *>(xs + col * 128 + 16 * k);
        }
    }
}

// ----------------------------------------------------------------------------- attention
__device__ __forceinline__ int fp8_first_masked_tile(int q0, int Nq, int Nk, int causal) {
    const int j_tail = Nk / 128;
    if (!causal) return j_tail;
    const int d1 = q0 + (Nk - Nq) + 1;
    return min(j_tail, d1 <= 0 ? 0 : d1 / 128);
}

__device__ __forceinline__ int fp8_tile_count(int q0, int Nq, int Nk, int causal) {
    if (q0 >= Nq) return 0;
    int kv_end = Nk;
    if (causal) kv_end = min(Nk, min(q0 + 128, Nq) + (Nk - Nq));
    return kv_end > 0 ? (kv_end + 127) / 128 : 0;
}

struct Fp8Row {
    float m, l, alpha;
    bool rescale;
};

// One step of this thread's row over one K/V tile: scores into registers, the
// mask, the exact max (m moves, and O is to be rescaled, when some row of the warp
// grew by more than kFp8RescaleThreshold), p * kappa = 2^(s*sl2 - m + log2 kappa)
// taken in one exponential, E4M3 of it written over the first 32 columns of the
// score buffer, and the row sum of p (the sum of p * kappa times 1/kappa).
// lk = log2 kappa, inv_kappa = 2^-lk.
template <bool MASKED>
__device__ __forceinline__ Fp8Row fp8_softmax_tile(uint32_t s_addr, int c0, int lim, float sl2, float lk,
                                                   float inv_kappa, float m, float l) {
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
    float mx[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) mx[e] = fmax3(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1]), -INFINITY);
#pragma unroll
    for (int c = 16; c < 128; c += 2)
        mx[(c >> 1) & 7] = fmax3(mx[(c >> 1) & 7], __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
    const float rmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
    // The scale factor sl2 is positive, so the max of the scaled scores is rmax * sl2.
    const float m_cand = fmaxf(m, rmax * sl2);
    Fp8Row r;
    r.alpha = 1.f;
    r.rescale = __any_sync(0xffffffffu, m_cand > m + kFp8RescaleThreshold);
    if (r.rescale) {
        const float m_new_d = (m_cand == -INFINITY) ? 0.f : m_cand;  // never subtract -inf from -inf
        r.alpha = ex2_approx(m - m_new_d);
        m = m_cand;
    }
    const float m_d = (m == -INFINITY) ? 0.f : m;
    const uint64_t scale2 = f2_make(sl2, sl2), shift2 = f2_make(lk - m_d, lk - m_d);
    uint64_t rs2[2] = {f2_make(0.f, 0.f), f2_make(0.f, 0.f)};
    uint32_t pk[32];
#pragma unroll
    for (int e = 0; e < 128; e += 4) {
        const float2 xa = f2_split(ffma2(f2_make(__uint_as_float(s[e]), __uint_as_float(s[e + 1])), scale2, shift2));
        const float2 xb = f2_split(ffma2(f2_make(__uint_as_float(s[e + 2]), __uint_as_float(s[e + 3])), scale2, shift2));
        const float a0 = ex2_approx(xa.x), a1 = ex2_approx(xa.y), b0 = ex2_approx(xb.x), b1 = ex2_approx(xb.y);
        rs2[0] = fadd2(rs2[0], f2_make(a0, a1));
        rs2[1] = fadd2(rs2[1], f2_make(b0, b1));
        pk[e >> 2] = pack_e4m3x4(a0, a1, b0, b1);
    }
    tmem_st_32x32b_x32(s_addr, pk);
    const float2 rsum = f2_split(fadd2(rs2[0], rs2[1]));
    r.m = m;
    r.l = l * r.alpha + (rsum.x + rsum.y) * inv_kappa;
    return r;
}

template <bool MASKED>
__device__ __noinline__ Fp8Row fp8_softmax_tile_out(uint32_t s_addr, int c0, int lim, float sl2, float lk,
                                                    float inv_kappa, float m, float l) {
    return fp8_softmax_tile<MASKED>(s_addr, c0, lim, sl2, lk, inv_kappa, m, l);
}

// O (32 rows of this warp, 128 columns) *= alpha.
__device__ __noinline__ void fp8_rescale_o(uint32_t o_addr, float alpha) {
    const uint64_t a2 = f2_make(alpha, alpha);
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
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

template <bool BF16>
__global__ void __launch_bounds__(kFp8Threads, 1)
    fa_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const Fp8FwdArgs args) {
    using C = Fp8Cfg;
    using PK = Pack<BF16>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sb = raw + pad;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int bh = blockIdx.y;
    const int mb = args.num_m - 1 - (int)blockIdx.x;  // heaviest causal row block first
    const int q0 = mb * 128;
    const int Nq = args.Nq, Nk = args.Nk, causal = args.causal;
    const int n = fp8_tile_count(q0, Nq, Nk, causal);
    const int jm = fp8_first_masked_tile(q0, Nq, Nk, causal);
    const int nbk = (Nk + 127) / 128;
    const float *ks = args.k_scale + (size_t)bh * nbk;
    const float *vs = args.v_scale + (size_t)bh * nbk;

    auto bar = [&](int idx) -> uint32_t { return sb + C::kOffBar + 8u * (uint32_t)idx; };
    constexpr int S_ = kFp8Stages;
    constexpr int B_QFULL = 0;
    auto B_KFULL = [](int s) { return 1 + s; };
    auto B_KEMPTY = [](int s) { return 1 + S_ + s; };
    auto B_VFULL = [](int s) { return 1 + 2 * S_ + s; };
    auto B_VEMPTY = [](int s) { return 1 + 3 * S_ + s; };
    auto B_SFULL = [](int b) { return 1 + 4 * S_ + b; };
    auto B_PFULL = [](int b) { return 4 + 4 * S_ + b; };
    auto B_PVDONE = [](int b) { return 7 + 4 * S_ + b; };
    constexpr int B_OFINAL = 10 + 4 * S_;
    auto B_MMAFIN = [](int w) { return 11 + 4 * S_ + w; };
    volatile uint32_t *tmem_holder = reinterpret_cast<volatile uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
    float *vmax_slot = reinterpret_cast<float *>(smem + C::kOffMisc + 8);
    int *status = args.status;

    if (threadIdx.x == 0) {
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
    }
    if (warp == 7) {
        // The largest V block scale of this head (kappa_j = 2^7 s_v(j) / max s_v <= 2^7).
        float vmx = 0.f;
        for (int j = lane; j < nbk; j += 32) vmx = fmaxf(vmx, __ldg(vs + j));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) vmx = fmaxf(vmx, __shfl_xor_sync(0xffffffffu, vmx, o));
        if (lane == 0) *vmax_slot = vmx;
    }
    if (warp == kFp8WarpPv) {
        tmem_alloc(sb + C::kOffMisc, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    constexpr uint32_t hi = sdesc_hi_sw128(1024);
    constexpr uint32_t idesc = idesc_e4m3(128, 128);

    if (warp == kFp8WarpTma) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && n > 0) {
            uint32_t pend_k = 0, pend_v = 0, par_k = 0, par_v = 0;
            mbar_arrive_expect_tx(bar(B_QFULL), C::kTileBytes);
            tma_load_3d(sb + C::kOffQ, &tmQ, 0, q0, bh, bar(B_QFULL));
            auto load = [&](bool is_v, int tile) -> bool {
                const int s = tile % S_;
                const uint32_t it = (uint32_t)(tile / S_);
                if (!mbar_wait_backoff(bar(is_v ? B_VEMPTY(s) : B_KEMPTY(s)), (it & 1u) ^ 1u, abort_flag, status, 64))
                    return false;
                const uint32_t full = bar(is_v ? B_VFULL(s) : B_KFULL(s));
                mbar_arrive_expect_tx(full, C::kTileBytes);
                if (is_v)  // V^T tile: x = first key (bytes), y = head-dim row
                    tma_load_3d(sb + C::kOffV + s * C::kTileBytes, &tmV, tile * 128, 0, bh, full);
                else
                    tma_load_3d(sb + C::kOffK + s * C::kTileBytes, &tmK, 0, tile * 128, bh, full);
                (is_v ? pend_v : pend_k) |= 1u << s;
                uint32_t &par = is_v ? par_v : par_k;
                par = (par & ~(1u << s)) | ((it & 1u) << s);
                return true;
            };
            bool ok = true;
            for (int t = 0; ok && t < min(n, 3); ++t) ok = load(false, t);
            for (int j = 0; ok && j < n; ++j) ok = load(true, j) && (j + 3 >= n || load(false, j + 3));
            volatile int no_abort = 0;
            mbar_wait_bounded(bar(B_QFULL), 0, &no_abort, status);
            for (int s = 0; s < S_; ++s) {
                if (pend_k & (1u << s)) mbar_wait_bounded(bar(B_KFULL(s)), (par_k >> s) & 1u, &no_abort, status);
                if (pend_v & (1u << s)) mbar_wait_bounded(bar(B_VFULL(s)), (par_v >> s) & 1u, &no_abort, status);
            }
        }
    } else if (warp == kFp8WarpS) {
        // ------------------------------------------------------------ MMA issuer: S stream
        if (lane == 0 && n > 0) {
            const uint32_t q_lo = sdesc_lo(sb + C::kOffQ, 16);
            const uint32_t k_lo = sdesc_lo(sb + C::kOffK, 16);
            bool ok = mbar_wait_bounded(bar(B_QFULL), 0, abort_flag, status);
            for (int t = 0; ok && t < n; ++t) {
                const int b = t % 3, s = t % S_;
                if (t >= 3) ok = mbar_wait_backoff(bar(B_PVDONE(b)), (uint32_t)(t / 3 - 1) & 1u, abort_flag, status, 64);
                ok = ok && mbar_wait_backoff(bar(B_KFULL(s)), (uint32_t)(t / S_) & 1u, abort_flag, status, 64);
                if (!ok) break;
                tc_fence_after();
                // S(t) = Q8 K8_t^T: 32 head-dim elements (32 bytes) per instruction.
                const uint32_t kt_lo = k_lo + (uint32_t)(s * (C::kTileBytes >> 4));
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    umma_ss_f8(tmem + C::tmem_s(b), q_lo + 2 * k, hi, kt_lo + 2 * k, hi, idesc, k > 0 ? 1u : 0u);
                umma_commit(bar(B_SFULL(b)));
                umma_commit(bar(B_KEMPTY(s)));
            }
            umma_commit(bar(B_MMAFIN(1)));
            volatile int no_abort = 0;
            mbar_wait_bounded(bar(B_MMAFIN(1)), 0, &no_abort, status);
        }
    } else if (warp == kFp8WarpPv) {
        // ------------------------------------------------------------ MMA issuer: PV stream
        if (lane == 0 && n > 0) {
            const uint32_t v_lo = sdesc_lo(sb + C::kOffV, 16);
            const uint32_t d_o = tmem + C::kTmemO;
            bool ok = true;
            for (int j = 0; ok && j < n; ++j) {
                const int b = j % 3, s = j % S_;
                ok = mbar_wait_backoff(bar(B_PFULL(b)), (uint32_t)(j / 3) & 1u, abort_flag, status, 32) &&
                     mbar_wait_backoff(bar(B_VFULL(s)), (uint32_t)(j / S_) & 1u, abort_flag, status, 32);
                if (!ok) break;
                tc_fence_after();
                // O += P8(j) V8_j: P8 from tensor memory (4 codes per column), V^T K-major,
                // 32 keys (32 bytes) per instruction.
                const uint32_t vt_lo = v_lo + (uint32_t)(s * (C::kTileBytes >> 4));
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    umma_ts_f8(d_o, tmem + C::tmem_s(b) + 8 * k, vt_lo + 2 * k, hi, idesc, (j > 0 || k > 0) ? 1u : 0u);
                umma_commit(bar(B_PVDONE(b)));
                umma_commit(bar(B_VEMPTY(s)));
            }
            if (ok) umma_commit(bar(B_OFINAL));
            umma_commit(bar(B_MMAFIN(0)));
            volatile int no_abort = 0;
            mbar_wait_bounded(bar(B_MMAFIN(0)), 0, &no_abort, status);
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ softmax / correction / epilogue
        const int i = q0 + warp * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        const uint32_t o_addr = lane_base + C::kTmemO;
        const int lim = causal ? min(i + (Nk - Nq), Nk - 1) : Nk - 1;
        const float vmax = *vmax_slot;
        const float inv_vmax = vmax > 0.f ? 1.f / vmax : 0.f;
        const float base = args.scale_log2 * __ldg(args.q_scale + (size_t)bh * args.num_m + mb);
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        float ks_next = n > 0 ? __ldg(ks) : 0.f, vs_next = n > 0 ? __ldg(vs) : 0.f;
        for (int j = 0; j < n; ++j) {
            const int b = j % 3;
            // kappa_j = 2^7 s_v(j) / max s_v, as its base-2 logarithm and the reciprocal
            // that undoes it in the row sum (the two agree to the rounding of one ex2).
            const float sl2 = base * ks_next;
            const float lk = 7.0f + __log2f(vs_next * inv_vmax);
            const float inv_kappa = ex2_approx(-lk);
            if (j + 1 < n) {
                ks_next = __ldg(ks + j + 1);
                vs_next = __ldg(vs + j + 1);
            }
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(B_SFULL(b)), (uint32_t)(j / 3) & 1u, abort_flag, status));
            if (!ok) break;
            tc_fence_after();
            const uint32_t s_addr = lane_base + C::tmem_s(b);
            const Fp8Row r = j >= jm ? fp8_softmax_tile_out<true>(s_addr, j * 128, lim, sl2, lk, inv_kappa, m, l)
                                     : fp8_softmax_tile<false>(s_addr, 0, 0, sl2, lk, inv_kappa, m, l);
            m = r.m;
            l = r.l;
            if (r.rescale && j > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(B_PVDONE((j - 1) % 3)), (uint32_t)((j - 1) / 3) & 1u,
                                                               abort_flag, status));
                if (!ok) break;
                tc_fence_after();
                fp8_rescale_o(o_addr, r.alpha);
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
        if (ok && __any_sync(0xffffffffu, i < Nq)) {
            // O = acc * (max s_v / 2^7) / l (0 for a row that saw no key), LSE = m ln2 + ln l.
            const bool valid = i < Nq;
            const float inv = (l > 0.f) ? (vmax / kFp8PScale) / l : 0.f;
            typename PK::T *orow_g = reinterpret_cast<typename PK::T *>(args.o) + ((size_t)bh * Nq + i) * 128;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
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
    if (warp == kFp8WarpPv) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

cudaError_t launch_fp8_quant(bool bf16, bool transpose, const Fp8QuantArgs &a, int BH, cudaStream_t stream) {
    const dim3 grid((unsigned)a.num_blocks, (unsigned)BH, 1);
    if (bf16)
        return transpose ? launch_kernel(fa_fp8_quant_kernel<true, true>, grid, dim3(256), 0, stream, a)
                         : launch_kernel(fa_fp8_quant_kernel<true, false>, grid, dim3(256), 0, stream, a);
    return transpose ? launch_kernel(fa_fp8_quant_kernel<false, true>, grid, dim3(256), 0, stream, a)
                     : launch_kernel(fa_fp8_quant_kernel<false, false>, grid, dim3(256), 0, stream, a);
}

cudaError_t launch_fwd_fp8(bool bf16_out, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           const Fp8FwdArgs &a, int BH, cudaStream_t stream) {
    auto kern = bf16_out ? fa_fwd_fp8_kernel<true> : fa_fwd_fp8_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Fp8Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, dim3((unsigned)a.num_m, (unsigned)BH, 1), dim3(kFp8Threads), Fp8Cfg::kSmemBytes,
                         stream, tq, tk, tv, a);
}

}  // namespace fa
