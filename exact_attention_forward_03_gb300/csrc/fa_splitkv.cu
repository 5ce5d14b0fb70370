// fa_splitkv.cu -- split-KV attention forward (flash-decoding) and the
// LSE-weighted combine, on CUDA cores.
//
// "02 · FA2: parallelism and work partitioning", §2: with one query row per
// (batch, head) the Q-block grid has only B*H CTAs, so the keys are cut into
// num_splits ranges; each range yields a partial (O_s, LSE_s) and a combine
// kernel merges them.  With Nq = 1 every key is read once, so the work is
// bound by HBM bandwidth; the dot products run on CUDA cores in fp32.
//
// Split kernel: one CTA of 128 threads per (split, query row, query head).  K/V
// tiles of 64 keys stream through a 3-stage ring of shared-memory slots,
// loaded by TMA with the 128-byte swizzle (row r's 16-byte chunk c sits at
// chunk c ^ (r & 7), so the row-per-thread reads below hit distinct banks).
//   scores:  thread t takes key t/2 and half t%2 of the head dimension,
//            q (pre-multiplied by scale*log2 e) in registers; the two halves
//            meet through one shuffle.
//   softmax: the tile max is reduced across the CTA; m, alpha and p follow
//            the online-softmax update in base 2; each thread keeps its own
//            share of l, reduced once at the end (the row sum is the only
//            cross-thread sum and it is deferred).
//   P V:     thread t owns output column t % d and every (128/d)-th key of
//            the tile; p comes from shared memory.
// Each partial is written normalised: O_s = O~_s / l_s, LSE_s = m_s ln 2 + ln l_s
// (O_s = 0, LSE_s = -inf for a split with no visible key).
#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {

constexpr int kSplitThreads = 128;

template <int D>
struct SplitCfg {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int kStages = 3;
    static constexpr int kBlocks = D / 64;
    static constexpr int kBlockBytes = kDecBc * 128;  // one 64-column block of a 64-key tile
    static constexpr int kTileBytes = kDecBc * D * 2;
    static constexpr int kStageBytes = 2 * kTileBytes;  // K then V
    static constexpr int kOffBar = kStages * kStageBytes;
    static constexpr int kOffP = kOffBar + kStages * 8;        // float p[2][64]
    static constexpr int kOffRed = kOffP + 2 * kDecBc * 4;     // float red[2][4]
    static constexpr int kOffOred = kOffRed + 2 * 4 * 4;       // float ored[128] (final reduce)
    static constexpr int kOffMisc = kOffOred + kSplitThreads * 4;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
    static constexpr int kKeyGroups = kSplitThreads / D;  // threads per output column in P V
};

template <int D, bool BF16>
__global__ void __launch_bounds__(kSplitThreads)
    fa_splitkv_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const SplitArgs a) {
    using C = SplitCfg<D>;
    using PK = Pack<BF16>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sb = raw + pad;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    // CTA order (fastest first): query head within its group, split, query row, K/V
    // head.  The CTAs of one group that read the same key range are launched side
    // by side and stream the same K/V tiles at the same time, so under grouped-query
    // attention all but one of them find the tiles in L2.
    const long long idx = blockIdx.x;
    const int hg = (int)(idx % a.group);
    long long rest = idx / a.group;
    const int split = (int)(rest % a.num_splits);
    rest /= a.num_splits;
    const int i = (int)(rest % a.Nq);
    const int kvh = (int)(rest / a.Nq);  // K/V head b*H_kv + h_kv
    const int H_kv = a.H / a.group;
    const int bh = (kvh / H_kv) * a.H + (kvh % H_kv) * a.group + hg;  // query head b*H + h_kv*group + hg
    const size_t out_row = (size_t)split * a.BH * a.Nq + (size_t)bh * a.Nq + i;

    const int k0 = split * a.split_len;
    int k1 = min(k0 + a.split_len, a.Nk);
    if (a.causal) k1 = min(k1, i + (a.Nk - a.Nq) + 1);
    if (k0 >= k1) {  // nothing visible in this split
        for (int t = tid; t < D; t += kSplitThreads) a.o_part[out_row * D + t] = 0.f;
        if (tid == 0) a.lse_part[out_row] = -INFINITY;
        return;
    }
    const int nt = (k1 - k0 + kDecBc - 1) / kDecBc;

    auto bar = [&](int s) -> uint32_t { return sb + C::kOffBar + 8u * (uint32_t)s; };
    float *p_s = reinterpret_cast<float *>(smem + C::kOffP);
    float *red = reinterpret_cast<float *>(smem + C::kOffRed);
    float *ored = reinterpret_cast<float *>(smem + C::kOffOred);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc);

    auto issue = [&](int t) {
        const int s = t % C::kStages;
        const uint32_t dst = sb + s * C::kStageBytes;
        const int y = k0 + t * kDecBc;
        mbar_arrive_expect_tx(bar(s), 2 * C::kTileBytes);
        for (int b = 0; b < C::kBlocks; ++b) {
            tma_load_3d(dst + b * C::kBlockBytes, &tmK, b * 64, y, kvh, bar(s));
            tma_load_3d(dst + C::kTileBytes + b * C::kBlockBytes, &tmV, b * 64, y, kvh, bar(s));
        }
    };

    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) mbar_init(bar(s), 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    __syncthreads();
    int issued = 0;
    if (tid == 0) {
        for (; issued < min(nt, C::kStages); ++issued) issue(issued);
    }

    // q for this thread's half of the head dimension, pre-scaled into base-2 units.
    const int kk = tid >> 1;  // key within the tile for the score phase
    const int half = tid & 1;
    constexpr int kChunks = D / 16;  // 16-byte chunks per half row
    float qf[D / 2];
    {
        const typename PK::T *qrow = reinterpret_cast<const typename PK::T *>(a.q) + ((size_t)bh * a.Nq + i) * D;
#pragma unroll
        for (int cc = 0; cc < kChunks; ++cc) {
            const uint4 u = *reinterpret_cast<const uint4 *>(qrow + (half * kChunks + cc) * 8);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = PK::unpack(w[e]);
                qf[cc * 8 + 2 * e] = f.x * a.scale_log2;
                qf[cc * 8 + 2 * e + 1] = f.y * a.scale_log2;
            }
        }
    }
    const int ocol = tid % D;       // output column owned in the P V phase
    const int kgrp = tid / D;       // key group (keys kgrp, kgrp + kKeyGroups, ...)
    const int oblk = ocol >> 6, ochunk = (ocol & 63) >> 3, opos = ocol & 7;
    float o_acc = 0.f;
    float m = -INFINITY, l_part = 0.f;

    for (int t = 0; t < nt; ++t) {
        const int s = t % C::kStages;
        const bool ok = mbar_wait_bounded(bar(s), (uint32_t)(t / C::kStages) & 1u, abort_flag, a.status);
        const uint8_t *ktile = smem + s * C::kStageBytes;
        float sc = 0.f;
        if (ok) {
#pragma unroll
            for (int cc = 0; cc < kChunks; ++cc) {
                const int g = half * kChunks + cc;  // 16-byte chunk index along the row
                const int blk = g >> 3, c = g & 7;
                const uint4 u =
                    *reinterpret_cast<const uint4 *>(ktile + blk * C::kBlockBytes + kk * 128 + ((c ^ (kk & 7)) << 4));
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = PK::unpack(w[e]);
                    sc = fmaf(qf[cc * 8 + 2 * e], f.x, sc);
                    sc = fmaf(qf[cc * 8 + 2 * e + 1], f.y, sc);
                }
            }
        }
        sc += __shfl_xor_sync(0xffffffffu, sc, 1);
        if (k0 + t * kDecBc + kk >= k1) sc = -INFINITY;
        float wm = sc;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
        if (lane == 0) red[(t & 1) * 4 + warp] = wm;
        if (__syncthreads_or(!ok)) {
            // A load never arrived: wait (bounded) for the ones in flight, then leave.
            if (tid == 0) {
                volatile int no_abort = 0;
                for (int u = t; u < issued; ++u)
                    mbar_wait_bounded(bar(u % C::kStages), (uint32_t)(u / C::kStages) & 1u, &no_abort, a.status);
            }
            return;
        }
        // Every thread has finished tile t-1: its slot can be refilled.
        if (tid == 0 && t >= 1 && issued < nt) issue(issued++);
        const float mx = fmaxf(fmaxf(red[(t & 1) * 4 + 0], red[(t & 1) * 4 + 1]),
                               fmaxf(red[(t & 1) * 4 + 2], red[(t & 1) * 4 + 3]));
        const float m_new = fmaxf(m, mx);
        const float m_d = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ex2_approx(m - m_d);
        const float p = ex2_approx(sc - m_d);
        if (half == 0) p_s[(t & 1) * kDecBc + kk] = p;
        l_part = l_part * alpha + (half == 0 ? p : 0.f);
        m = m_new;
        __syncthreads();
        const uint8_t *vtile = ktile + C::kTileBytes;
        const float *pt = p_s + (t & 1) * kDecBc;
        float acc = o_acc * alpha;
#pragma unroll 8
        for (int key = kgrp; key < kDecBc; key += C::kKeyGroups) {
            const uint16_t raw16 = *reinterpret_cast<const uint16_t *>(
                vtile + oblk * C::kBlockBytes + key * 128 + ((ochunk ^ (key & 7)) << 4) + opos * 2);
            const float vf = PK::unpack((uint32_t)raw16).x;
            acc = fmaf(pt[key], vf, acc);
        }
        o_acc = acc;
    }

    // Deferred reductions: l over all threads, O over the key groups.
    float lw = l_part;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
    __syncthreads();  // red / p_s of the last tile are no longer read
    if (lane == 0) red[warp] = lw;
    ored[tid] = o_acc;
    __syncthreads();
    const float l = red[0] + red[1] + red[2] + red[3];
    if (tid < D) {
        float o = 0.f;
#pragma unroll
        for (int g = 0; g < C::kKeyGroups; ++g) o += ored[g * D + tid];
        a.o_part[out_row * D + tid] = (l > 0.f) ? o / l : 0.f;
    }
    if (tid == 0) {
        const float m_d = (m == -INFINITY) ? 0.f : m;
        a.lse_part[out_row] = (l > 0.f) ? m_d * 0.69314718055994531f + logf(l) : -INFINITY;
    }
}

// Combine: one warp per row; lane t owns d/32 consecutive output columns.
template <int D, bool BF16>
__global__ void __launch_bounds__(128) fa_combine_kernel(const CombineArgs a) {
    using PK = Pack<BF16>;
    constexpr int kPer = D / 32;
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (row >= a.rows) return;
    const int S = a.num_splits;
    float M = -INFINITY;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, a.lse_part[(size_t)s * a.rows + row]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
    float wsum = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < S; ++s) {
            const float ls = a.lse_part[(size_t)s * a.rows + row];
            const float w = (ls == -INFINITY) ? 0.f : expf(ls - M);
            wsum += w;
            const float *op = a.o_part + ((size_t)s * a.rows + row) * D + lane * kPer;
            if constexpr (kPer == 4) {
                const float4 v = *reinterpret_cast<const float4 *>(op);
                acc[0] = fmaf(w, v.x, acc[0]);
                acc[1] = fmaf(w, v.y, acc[1]);
                acc[2] = fmaf(w, v.z, acc[2]);
                acc[3] = fmaf(w, v.w, acc[3]);
            } else {
                const float2 v = *reinterpret_cast<const float2 *>(op);
                acc[0] = fmaf(w, v.x, acc[0]);
                acc[1] = fmaf(w, v.y, acc[1]);
            }
        }
    }
    const float inv = (wsum > 0.f) ? 1.f / wsum : 0.f;
    typename PK::T *orow = reinterpret_cast<typename PK::T *>(a.o) + (size_t)row * D + lane * kPer;
    if constexpr (kPer == 4) {
        uint2 u;
        u.x = PK::pack(acc[0] * inv, acc[1] * inv);
        u.y = PK::pack(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2 *>(orow) = u;
    } else {
        *reinterpret_cast<uint32_t *>(orow) = PK::pack(acc[0] * inv, acc[1] * inv);
    }
    if (lane == 0 && a.lse != nullptr) a.lse[row] = (wsum > 0.f) ? M + logf(wsum) : -INFINITY;
}

template <int D, bool BF16>
static cudaError_t launch_splitkv_t(const CUtensorMap &tk, const CUtensorMap &tv, const SplitArgs &a,
                                    cudaStream_t stream) {
    using C = SplitCfg<D>;
    auto kern = fa_splitkv_kernel<D, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const long long ctas = (long long)a.num_splits * a.Nq * a.BH;
    return launch_kernel(kern, dim3((unsigned)ctas), dim3(kSplitThreads), C::kSmemBytes, stream, tk, tv, a);
}

cudaError_t launch_splitkv(int d, bool bf16, const CUtensorMap &tk, const CUtensorMap &tv, const SplitArgs &a,
                           cudaStream_t stream) {
    if (d == 64) return bf16 ? launch_splitkv_t<64, true>(tk, tv, a, stream)
                             : launch_splitkv_t<64, false>(tk, tv, a, stream);
    return bf16 ? launch_splitkv_t<128, true>(tk, tv, a, stream) : launch_splitkv_t<128, false>(tk, tv, a, stream);
}

template <int D, bool BF16>
static cudaError_t launch_combine_t(const CombineArgs &a, cudaStream_t stream) {
    const long long blocks = (a.rows + 3) / 4;
    return launch_kernel(fa_combine_kernel<D, BF16>, dim3((unsigned)blocks), dim3(128), 0, stream, a);
}

cudaError_t launch_combine(int d, bool bf16, const CombineArgs &a, cudaStream_t stream) {
    if (d == 64) return bf16 ? launch_combine_t<64, true>(a, stream) : launch_combine_t<64, false>(a, stream);
    return bf16 ? launch_combine_t<128, true>(a, stream) : launch_combine_t<128, false>(a, stream);
}

}  // namespace fa
