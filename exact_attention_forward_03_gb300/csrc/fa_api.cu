// fa_api.cu -- the C ABI declared in include/fa.h: argument checks, TMA
// tensor-map encoding, split planning and kernel launches.  Host code only;
// the kernels live in fa_fwd_sm103.cu and fa_splitkv.cu.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdio>
#include <cstdint>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace fa {

// Per-device status word: kernels OR error bits into it (see kDevErrTimeout).
__device__ int g_status_word;

// Built-in scratch for fa_fwd_splitkv_noalloc: the split partials live here
// instead of in a caller-provided workspace.  Every GPU that loads this library
// holds these bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_splitkv_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int *status = nullptr;  // device address of g_status_word
    int num_sms = 0;
    // fa_fwd_host: copy-in and copy-out streams and the events that order them
    // against the caller's stream, created on first use; host_mu serialises the
    // enqueueing of calls that share them.
    bool host_ready = false;
    cudaStream_t copy_in = nullptr, copy_out = nullptr;
    cudaEvent_t ev_entry = nullptr, ev_in = nullptr, ev_comp = nullptr, ev_exit = nullptr;
    std::mutex host_mu;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
void *g_scratch_addr[kMaxDevices];  // device address of g_splitkv_scratch, looked up once per device
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Why the calling thread last got FA_ERR_CUDA (read by fa_last_error).
thread_local char t_last_error[160];

int cuda_fail(const char *where, int code, const char *name) {
    snprintf(t_last_error, sizeof(t_last_error), "%s failed: %s (%d)", where, name ? name : "CUresult", code);
    return FA_ERR_CUDA;
}
int cuda_fail(const char *where, cudaError_t e) { return cuda_fail(where, (int)e, cudaGetErrorName(e)); }
int launch_status(const char *what, cudaError_t e) { return e == cudaSuccess ? FA_OK : cuda_fail(what, e); }

int dev_state(DeviceState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
    if (dev < 0 || dev >= kMaxDevices) return cuda_fail("device index", dev, "out of range");
    // The tensor-map encoder is a driver call and needs a current context; a thread
    // that has made no runtime call yet (an autograd worker, say) has none.  Setting
    // the device once per thread makes its primary context current.
    thread_local int t_ctx_dev = -1;
    if (t_ctx_dev != dev) {
        if ((e = cudaSetDevice(dev)) != cudaSuccess) return cuda_fail("cudaSetDevice", e);
        t_ctx_dev = dev;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &st = g_dev[dev];
    if (!st.ready) {
        void *p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_status_word)) != cudaSuccess) return cuda_fail("cudaGetSymbolAddress", e);
        int sms = 0;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail("cudaDeviceGetAttribute", e);
        st.status = static_cast<int *>(p);
        st.num_sms = sms;
        st.ready = true;
    }
    if (g_encode == nullptr) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return cuda_fail("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)", (int)q, "no entry point");
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *out = &st;
    return FA_OK;
}

// [BH][rows][d] 16-bit tensor, boxes of 64 columns (128 bytes) x box_rows rows x 1 head,
// 128-byte swizzle; rows beyond `rows` read as zero.
int make_map(CUtensorMap *map, const void *ptr, bool bf16, int d, int rows, int BH, int box_rows) {
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)rows * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                          const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : cuda_fail("cuTensorMapEncodeTiled", (int)r, nullptr);
}

// Packed [tokens][heads][d] 16-bit tensor of a variable-length batch: boxes of 64
// columns x 1 head x box_rows tokens (the same 128-byte rows in shared memory as
// make_map's boxes), 128-byte swizzle; tokens beyond `tokens` read as zero.
int make_map_packed(CUtensorMap *map, const void *ptr, bool bf16, int d, int heads, int tokens, int box_rows) {
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                          const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : cuda_fail("cuTensorMapEncodeTiled", (int)r, nullptr);
}

// 8-bit tensor [heads][rows][cols] (cols a multiple of 16), boxes of 128 columns x
// 128 rows x 1 head, 128-byte swizzle; rows and columns past the end read as zero.
int make_map_u8(CUtensorMap *map, const void *ptr, int cols, int rows, int heads) {
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)cols, (cuuint64_t)rows * cols};
    cuuint32_t box[3] = {128, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : cuda_fail("cuTensorMapEncodeTiled", (int)r, nullptr);
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_common(const void *q, const void *k, const void *v, const void *o, const float *lse, int B, int H,
                 int Nq, int Nk, int d, int causal, float scale, int dtype) {
    if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return FA_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0) return FA_ERR_INVALID_ARG;
    if ((long long)B * H > INT32_MAX) return FA_ERR_INVALID_ARG;
    if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16)) return FA_ERR_MISALIGNED;
    if (lse != nullptr && !aligned(lse, 4)) return FA_ERR_MISALIGNED;
    return FA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Heads whose row blocks the forward's launch order interleaves (FwdArgs::head_group).
// Only a causal grid of at most about eight waves (ctas <= 8 x SMs) gains from it: its
// heavy last row blocks then no longer start at the end of the launch (measured on
// GB300: +9.6 % at B4 H16 N1024 causal, 11-29 % on the same grids run two CTAs per SM;
// 1-2 % lost on the 27-wave causal B2 H32 N8192 launch, 1-4 % on a packed batch).
// Without a mask every row block costs the same and the wider K/V working set only
// costs (B4 H16 N1024: -0.6 % with one CTA per SM, -3.5 % with two).  As many heads as
// keep their K and V, kv_bytes per head, within about 32 MiB of L2, at most 16 and at
// most the grid's heads; 1 (the plain order) otherwise.
int fwd_head_group(double kv_bytes, int heads, long long ctas, int num_sms, int causal) {
    if (!causal || ctas > 8LL * num_sms) return 1;
    int g = kv_bytes > 0 ? (int)(32.0 * 1024 * 1024 / kv_bytes) : 16;
    g = g < 1 ? 1 : (g > 16 ? 16 : g);
    return g < heads ? g : heads;
}

// Whether the d = 64 forward runs in its two-CTAs-per-SM form (one score buffer per
// CTA, so each CTA's S -> softmax -> PV chain is serial, but one CTA's set-up, last
// GEMM and epilogue overlap the other's tile loop).  That pays only where those fixed
// costs weigh most: grids of three to eight waves whose CTAs visit at most 16 K/V
// tiles.  Measured on GB300 (paired vs. one CTA per SM, 50 calls between events): B4
// H16 N1024 f16 +3.7 % (+7.2 % causal), B4 H32 N1024 +0.8 % (+21 % causal), B2 H16
// N2048 causal +15 %, B3 H16 N2048 causal +4.0 % (non-causal +1.8 % once neither form
// interleaves heads); lost at under two waves (-6 to -19 %), on longer rows (B2 H16
// N4096 -17 % non-causal) and on large grids (B2 H32 N8192 -9 % causal, -13 %
// non-causal).
bool fwd_pair(int d, int Nk, long long ctas, int num_sms) {
    const int tiles = (Nk + kFwdBc - 1) / kFwdBc;
    return d == 64 && ctas >= 3LL * num_sms && ctas <= 8LL * num_sms && tiles <= 16;
}

int auto_splits(int num_sms, long long rows, int Nk) {
    // About 48 CTAs per SM, at least one 64-key tile per split, at most 64 splits.
    // Measured on GB300 at B=32, H=32, Nk=16384, d=128 (GB/s of compulsory bytes by
    // split count): 1: 5802, 2: 6580, 3: 6365, 4: 6585, 6: 6600, 8: 6701, 12: 6616,
    // 16: 6554, 32: 6233; this target picks 8 there.
    const long long target = 48LL * (num_sms > 0 ? num_sms : 148);
    long long s = (target + rows - 1) / rows;
    const long long tiles = (Nk + kDecBc - 1) / kDecBc;
    if (s > tiles) s = tiles;
    if (s > 64) s = 64;
    if (s < 1) s = 1;
    return (int)s;
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

int fa_version(void) { return 100; }

const char *fa_last_error(void) { return t_last_error; }

const char *fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "ok";
        case FA_ERR_INVALID_ARG: return "invalid argument";
        case FA_ERR_UNSUPPORTED: return "unsupported head dimension (d must be 64 or 128)";
        case FA_ERR_MISALIGNED: return "misaligned pointer (16-byte alignment required)";
        case FA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case FA_ERR_CUDA: return "CUDA runtime error";
        case FA_ERR_DEVICE_TIMEOUT: return "a device-side bounded wait ran out";
        case FA_ERR_SCRATCH_LIMIT: return "split partials exceed the built-in 16 MiB scratch of fa_fwd_splitkv_noalloc";
        default: return "unknown status";
    }
}

int fa_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int H_kv, int Nq,
               int Nk, int d, int causal, float scale, fa_dtype dtype, fa_stream_t stream) {
    int rc = check_common(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale, dtype);
    if (rc != FA_OK) return rc;
    if (H_kv <= 0 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    int group = H / H_kv;
    if (group > 1 && (causal == 0 || Nq == 1) && (long long)group * Nq <= INT32_MAX) {
        // The `group` query heads of one K/V head are consecutive in q, o and lse, so they
        // form a single head of group*Nq query rows against that K/V head.  Without a
        // causal mask (and with one query row, which sees every key) the rows need not
        // know which head they came from: run that problem, which reads each K/V tile once
        // for the whole group.
        H = H_kv;
        Nq *= group;
        causal = 0;
        group = 1;
    }
    const int num_m = (Nq + kFwdTilesPerCta * kFwdBr - 1) / (kFwdTilesPerCta * kFwdBr);
    if (B * H > 65535) return FA_ERR_INVALID_ARG;  // grid.y limit
    DeviceState *st = nullptr;
    if ((rc = dev_state(&st)) != FA_OK) return rc;
    const bool bf16 = dtype == FA_BF16;
    const int BH = B * H;
    CUtensorMap tq, tk, tv, to;
    if (make_map(&tq, q, bf16, d, Nq, BH, kFwdBr) != FA_OK || make_map(&tk, k, bf16, d, Nk, B * H_kv, kFwdBc) != FA_OK ||
        make_map(&tv, v, bf16, d, Nk, B * H_kv, kFwdBc) != FA_OK || make_map(&to, o, bf16, d, Nq, BH, kFwdBr) != FA_OK)
        return FA_ERR_CUDA;
    FwdArgs a;
    a.o = o;
    a.lse = lse;
    a.status = st->status;
    a.Nq = Nq;
    a.Nk = Nk;
    a.num_m = num_m;
    a.H = H;
    a.group = group;
    a.head_group = fwd_head_group(4.0 * Nk * d / group, BH, (long long)num_m * BH, st->num_sms, causal);
    a.cu_q = nullptr;
    a.cu_k = nullptr;
    a.total_q = 0;
    a.work = nullptr;
    a.num_seqs = 0;
    a.causal = causal;
    a.scale_log2 = scale * 1.4426950408889634f;
    const bool pair = fwd_pair(d, Nk, (long long)num_m * BH, st->num_sms);
    cudaError_t e = launch_fwd(d, bf16, tq, tk, tv, to, a, BH, reinterpret_cast<cudaStream_t>(stream), pair);
    return launch_status("kernel launch", e);
}

size_t fa_fwd_host_workspace_bytes(int B, int H, int H_kv, int Nq, int Nk, int d) {
    if (B <= 0 || H <= 0 || H_kv <= 0 || H % H_kv != 0 || Nq <= 0 || Nk <= 0 || (d != 64 && d != 128)) return 0;
    const size_t qb = (size_t)B * H * Nq * d * 2, kb = (size_t)B * H_kv * Nk * d * 2;
    return 2 * align256(qb) + 2 * align256(kb) + align256((size_t)B * H * Nq * sizeof(float));
}

int fa_fwd_host(const void *q_host, const void *k_host, const void *v_host, void *o_host, float *lse_host, int B,
                int H, int H_kv, int Nq, int Nk, int d, int causal, float scale, fa_dtype dtype, int num_chunks,
                void *workspace, size_t workspace_bytes, fa_stream_t stream) {
    if (q_host == nullptr || k_host == nullptr || v_host == nullptr || o_host == nullptr) return FA_ERR_INVALID_ARG;
    // The checks of fa_fwd_gqa on stand-in device pointers (the workspace's are only known below).
    const void *probe = reinterpret_cast<const void *>((uintptr_t)256);
    int rc = check_common(probe, probe, probe, probe, nullptr, B, H, Nq, Nk, d, causal, scale, dtype);
    if (rc != FA_OK) return rc;
    if (H_kv <= 0 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    const size_t need = fa_fwd_host_workspace_bytes(B, H, H_kv, Nq, Nk, d);
    if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < need) return FA_ERR_WORKSPACE;
    DeviceState *st = nullptr;
    if ((rc = dev_state(&st)) != FA_OK) return rc;
    std::lock_guard<std::mutex> lk(st->host_mu);
    cudaError_t e;
    if (!st->host_ready) {
        if ((e = cudaStreamCreateWithFlags(&st->copy_in, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&st->copy_out, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&st->ev_entry, cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&st->ev_in, cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&st->ev_comp, cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&st->ev_exit, cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail("fa_fwd_host stream setup", e);
        st->host_ready = true;
    }
    const int group = H / H_kv;
    const int kv_heads = B * H_kv;
    int chunks = num_chunks > 0 ? num_chunks : 8;
    if (chunks > kv_heads) chunks = kv_heads;
    const size_t q_head = (size_t)Nq * d * 2, k_head = (size_t)Nk * d * 2;  // bytes per head
    char *ws = static_cast<char *>(workspace);
    char *qd = ws;
    char *od = qd + align256((size_t)B * H * q_head);
    char *kd = od + align256((size_t)B * H * q_head);
    char *vd = kd + align256((size_t)kv_heads * k_head);
    float *ld = reinterpret_cast<float *>(vd + align256((size_t)kv_heads * k_head));
    const char *qh = static_cast<const char *>(q_host), *kh = static_cast<const char *>(k_host),
               *vh = static_cast<const char *>(v_host);
    char *oh = static_cast<char *>(o_host);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const auto h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
    // On an error after copies were queued, `stream` is still made to wait for them,
    // so that a caller who synchronises it may free the buffers.
    auto join = [&]() {
        if (cudaEventRecord(st->ev_in, st->copy_in) == cudaSuccess) cudaStreamWaitEvent(cs, st->ev_in, 0);
        if (cudaEventRecord(st->ev_exit, st->copy_out) == cudaSuccess) cudaStreamWaitEvent(cs, st->ev_exit, 0);
    };
    auto join_and_fail = [&](const char *what, cudaError_t err) {
        join();
        return cuda_fail(what, err);
    };
    if ((e = cudaEventRecord(st->ev_entry, cs)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(st->copy_in, st->ev_entry, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(st->copy_out, st->ev_entry, 0)) != cudaSuccess)
        return join_and_fail("fa_fwd_host ordering", e);
    // Chunk c covers K/V heads [bound(c), bound(c+1)).  The copies of all chunks stream
    // back to back; after the last chunk's inputs arrive only its compute and its output
    // copy remain, so the last two chunks are tapered to 1/2 and 1/4 of the others
    // (weights 1, ..., 1, 1/2, 1/4, in quarters), every chunk keeping at least one head.
    const long long w_total = chunks >= 4 ? 4LL * (chunks - 2) + 3 : chunks;
    auto bound = [&](int c) -> int {
        long long w = c;  // equal chunks
        if (chunks >= 4) w = c <= chunks - 2 ? 4LL * c : 4LL * (chunks - 2) + 2;
        if (chunks >= 4 && c == chunks) w = w_total;
        const int h = (int)((long long)kv_heads * w / w_total);
        return c == 0 ? 0 : (h < c ? c : (h > kv_heads - (chunks - c) ? kv_heads - (chunks - c) : h));
    };
    for (int c = 0; c < chunks; ++c) {
        // K/V heads [h0, h1) and their query heads [h0 * group, h1 * group)
        const int h0 = bound(c), h1 = bound(c + 1);
        const size_t qo = (size_t)h0 * group * q_head, qn = (size_t)(h1 - h0) * group * q_head;
        const size_t ko = (size_t)h0 * k_head, kn = (size_t)(h1 - h0) * k_head;
        const size_t lo = (size_t)h0 * group * Nq, ln = (size_t)(h1 - h0) * group * Nq;  // lse elements
        if ((e = cudaMemcpyAsync(qd + qo, qh + qo, qn, h2d, st->copy_in)) != cudaSuccess ||
            (e = cudaMemcpyAsync(kd + ko, kh + ko, kn, h2d, st->copy_in)) != cudaSuccess ||
            (e = cudaMemcpyAsync(vd + ko, vh + ko, kn, h2d, st->copy_in)) != cudaSuccess ||
            (e = cudaEventRecord(st->ev_in, st->copy_in)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(cs, st->ev_in, 0)) != cudaSuccess)
            return join_and_fail("fa_fwd_host copy in", e);
        rc = fa_fwd_gqa(qd + qo, kd + ko, vd + ko, od + qo, ld + lo, 1, (h1 - h0) * group, h1 - h0, Nq, Nk, d, causal,
                        scale, dtype, stream);
        if (rc != FA_OK) {
            join();
            return rc;
        }
        if ((e = cudaEventRecord(st->ev_comp, cs)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(st->copy_out, st->ev_comp, 0)) != cudaSuccess ||
            (e = cudaMemcpyAsync(oh + qo, od + qo, qn, d2h, st->copy_out)) != cudaSuccess ||
            (lse_host != nullptr &&
             (e = cudaMemcpyAsync(lse_host + lo, ld + lo, ln * sizeof(float), d2h, st->copy_out)) != cudaSuccess))
            return join_and_fail("fa_fwd_host copy out", e);
    }
    if ((e = cudaEventRecord(st->ev_exit, st->copy_out)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(cs, st->ev_exit, 0)) != cudaSuccess)
        return join_and_fail("fa_fwd_host ordering", e);
    return FA_OK;
}

int fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse, const int *cu_seqlens_q,
                  const int *cu_seqlens_k, int num_seqs, int max_seqlen_q, int total_q, int total_k, int H, int H_kv,
                  int d, int causal, float scale, fa_dtype dtype, fa_stream_t stream) {
    // The common checks with one "sequence" of the totals stand in for B, Nq, Nk.
    int rc = check_common(q, k, v, o, lse, 1, H, total_q, total_k, d, causal, scale, dtype);
    if (rc != FA_OK) return rc;
    if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr) return FA_ERR_INVALID_ARG;
    if (!aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4)) return FA_ERR_MISALIGNED;
    if (num_seqs <= 0 || max_seqlen_q <= 0 || max_seqlen_q > total_q) return FA_ERR_INVALID_ARG;
    if (H_kv <= 0 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if ((long long)num_seqs * H > 65535) return FA_ERR_INVALID_ARG;  // grid.y limit
    DeviceState *st = nullptr;
    if ((rc = dev_state(&st)) != FA_OK) return rc;
    const bool bf16 = dtype == FA_BF16;
    CUtensorMap tq, tk, tv, to;
    if (make_map_packed(&tq, q, bf16, d, H, total_q, kFwdBr) != FA_OK ||
        make_map_packed(&tk, k, bf16, d, H_kv, total_k, kFwdBc) != FA_OK ||
        make_map_packed(&tv, v, bf16, d, H_kv, total_k, kFwdBc) != FA_OK ||
        make_map_packed(&to, o, bf16, d, H, total_q, kFwdBr) != FA_OK)
        return FA_ERR_CUDA;
    FwdArgs a;
    a.o = o;
    a.lse = lse;
    a.status = st->status;
    a.Nq = 0;
    a.Nk = 0;
    a.num_m = (max_seqlen_q + kFwdBr - 1) / kFwdBr;
    a.H = H;
    a.group = H / H_kv;
    a.head_group = 1;
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    a.total_q = total_q;
    a.work = nullptr;
    a.num_seqs = num_seqs;
    a.causal = causal;
    a.scale_log2 = scale * 1.4426950408889634f;
    cudaError_t e = launch_fwd_varlen(d, bf16, tq, tk, tv, to, a, num_seqs, reinterpret_cast<cudaStream_t>(stream));
    return launch_status("kernel launch", e);
}

size_t fa_fwd_varlen_workspace_bytes(int num_seqs, int total_q) {
    if (num_seqs <= 0 || total_q <= 0) return 0;
    return 16 + 8 * ((size_t)(total_q + kFwdBr - 1) / kFwdBr + (size_t)num_seqs);
}

int fa_fwd_varlen_ws(const void *q, const void *k, const void *v, void *o, float *lse, const int *cu_seqlens_q,
                     const int *cu_seqlens_k, int num_seqs, int total_q, int total_k, int H, int H_kv, int d,
                     int causal, float scale, fa_dtype dtype, void *workspace, size_t workspace_bytes,
                     fa_stream_t stream) {
    int rc = check_common(q, k, v, o, lse, 1, H, total_q, total_k, d, causal, scale, dtype);
    if (rc != FA_OK) return rc;
    if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr) return FA_ERR_INVALID_ARG;
    if (!aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4)) return FA_ERR_MISALIGNED;
    if (num_seqs <= 0 || H_kv <= 0 || H % H_kv != 0 || H > 65535) return FA_ERR_INVALID_ARG;
    const long long capacity = (long long)(total_q + kFwdBr - 1) / kFwdBr + num_seqs;
    if (capacity > INT_MAX) return FA_ERR_INVALID_ARG;
    const size_t need = fa_fwd_varlen_workspace_bytes(num_seqs, total_q);
    if (workspace == nullptr || !aligned(workspace, 16) || workspace_bytes < need) return FA_ERR_WORKSPACE;
    DeviceState *st = nullptr;
    if ((rc = dev_state(&st)) != FA_OK) return rc;
    const bool bf16 = dtype == FA_BF16;
    CUtensorMap tq, tk, tv, to;
    if (make_map_packed(&tq, q, bf16, d, H, total_q, kFwdBr) != FA_OK ||
        make_map_packed(&tk, k, bf16, d, H_kv, total_k, kFwdBc) != FA_OK ||
        make_map_packed(&tv, v, bf16, d, H_kv, total_k, kFwdBc) != FA_OK ||
        make_map_packed(&to, o, bf16, d, H, total_q, kFwdBr) != FA_OK)
        return FA_ERR_CUDA;
    FwdArgs a;
    a.o = o;
    a.lse = lse;
    a.status = st->status;
    a.Nq = 0;
    a.Nk = 0;
    a.num_m = (int)capacity;
    a.H = H;
    a.group = H / H_kv;
    a.head_group = 1;
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    a.total_q = total_q;
    a.work = nullptr;
    a.num_seqs = num_seqs;
    a.causal = causal;
    a.scale_log2 = scale * 1.4426950408889634f;
    cudaError_t e = launch_fwd_varlen_planned(d, bf16, tq, tk, tv, to, a, static_cast<int *>(workspace), (int)capacity,
                                              reinterpret_cast<cudaStream_t>(stream));
    return launch_status("kernel launch", e);
}

int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int Nq, int Nk, int d,
           int causal, float scale, fa_dtype dtype, fa_stream_t stream) {
    return fa_fwd_gqa(q, k, v, o, lse, B, H, H, Nq, Nk, d, causal, scale, dtype, stream);
}

int fa_splitkv_num_splits(int B, int H, int Nq, int Nk, int d) {
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || (d != 64 && d != 128)) return 0;
    DeviceState *st = nullptr;
    int sms = 148;
    if (dev_state(&st) == FA_OK) sms = st->num_sms;
    return auto_splits(sms, (long long)B * H * Nq, Nk);
}

int fa_splitkv_split_len(int Nk, int num_splits) {
    if (Nk <= 0 || num_splits <= 0) return 0;
    const int tiles = (Nk + kDecBc - 1) / kDecBc;
    const int per = (tiles + num_splits - 1) / num_splits;
    return per * kDecBc;
}

size_t fa_splitkv_workspace_bytes(int B, int H, int Nq, int Nk, int d, int num_splits) {
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || (d != 64 && d != 128)) return 0;
    if (num_splits <= 0) num_splits = fa_splitkv_num_splits(B, H, Nq, Nk, d);
    if (num_splits <= 0 || num_splits > kMaxSplits) return 0;
    const size_t rows = (size_t)B * H * Nq;
    return align256((size_t)num_splits * rows * d * sizeof(float)) + align256((size_t)num_splits * rows * sizeof(float));
}

int fa_splitkv_combine(const float *o_part, const float *lse_part, void *o, float *lse, int num_splits, int B, int H,
                       int Nq, int d, fa_dtype dtype, fa_stream_t stream) {
    if (o_part == nullptr || lse_part == nullptr || o == nullptr) return FA_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || Nq <= 0 || num_splits <= 0 || num_splits > kMaxSplits) return FA_ERR_INVALID_ARG;
    if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!aligned(o_part, 16) || !aligned(o, 16) || !aligned(lse_part, 4)) return FA_ERR_MISALIGNED;
    if (lse != nullptr && !aligned(lse, 4)) return FA_ERR_MISALIGNED;
    const long long rows = (long long)B * H * Nq;
    if ((rows + 3) / 4 > INT32_MAX) return FA_ERR_INVALID_ARG;
    CombineArgs a;
    a.o_part = o_part;
    a.lse_part = lse_part;
    a.o = o;
    a.lse = lse;
    a.num_splits = num_splits;
    a.rows = rows;
    cudaError_t e = launch_combine(d, dtype == FA_BF16, a, reinterpret_cast<cudaStream_t>(stream));
    return launch_status("kernel launch", e);
}

int fa_fwd_splitkv_gqa(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int H_kv,
                       int Nq, int Nk, int d, int causal, float scale, fa_dtype dtype, int num_splits, void *workspace,
                       size_t workspace_bytes, fa_stream_t stream) {
    int rc = check_common(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale, dtype);
    if (rc != FA_OK) return rc;
    if (H_kv <= 0 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (num_splits > kMaxSplits) return FA_ERR_INVALID_ARG;
    DeviceState *st = nullptr;
    if ((rc = dev_state(&st)) != FA_OK) return rc;
    const long long rows = (long long)B * H * Nq;
    if (num_splits <= 0) num_splits = auto_splits(st->num_sms, rows, Nk);
    if ((long long)num_splits * rows > INT32_MAX) return FA_ERR_INVALID_ARG;
    const size_t need = fa_splitkv_workspace_bytes(B, H, Nq, Nk, d, num_splits);
    if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < need) return FA_ERR_WORKSPACE;
    const bool bf16 = dtype == FA_BF16;
    CUtensorMap tk, tv;
    if (make_map(&tk, k, bf16, d, Nk, B * H_kv, kDecBc) != FA_OK || make_map(&tv, v, bf16, d, Nk, B * H_kv, kDecBc) != FA_OK)
        return FA_ERR_CUDA;
    float *o_part = static_cast<float *>(workspace);
    float *lse_part =
        reinterpret_cast<float *>(static_cast<char *>(workspace) + align256((size_t)num_splits * rows * d * sizeof(float)));
    SplitArgs a;
    a.q = q;
    a.o_part = o_part;
    a.lse_part = lse_part;
    a.status = st->status;
    a.Nq = Nq;
    a.Nk = Nk;
    a.BH = B * H;
    a.H = H;
    a.group = H / H_kv;
    a.num_splits = num_splits;
    a.split_len = fa_splitkv_split_len(Nk, num_splits);
    a.causal = causal;
    a.scale_log2 = scale * 1.4426950408889634f;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = launch_splitkv(d, bf16, tk, tv, a, s);
    if (e != cudaSuccess) return cuda_fail("kernel launch", e);
    return fa_splitkv_combine(o_part, lse_part, o, lse, num_splits, B, H, Nq, d, dtype, stream);
}

int fa_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int Nq, int Nk,
                   int d, int causal, float scale, fa_dtype dtype, int num_splits, void *workspace,
                   size_t workspace_bytes, fa_stream_t stream) {
    return fa_fwd_splitkv_gqa(q, k, v, o, lse, B, H, H, Nq, Nk, d, causal, scale, dtype, num_splits, workspace,
                              workspace_bytes, stream);
}

int fa_fp8_quantize(const void *x, void *x8, float *scales, int BH, int N, int d, int transpose, fa_dtype dtype,
                    fa_stream_t stream) {
    if (x == nullptr || x8 == nullptr || scales == nullptr) return FA_ERR_INVALID_ARG;
    if (BH <= 0 || BH > 65535 || N <= 0 || (transpose != 0 && transpose != 1)) return FA_ERR_INVALID_ARG;
    if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
    if (d != 128) return FA_ERR_UNSUPPORTED;
    if (!aligned(x, 16) || !aligned(x8, 16) || !aligned(scales, 4)) return FA_ERR_MISALIGNED;
    DeviceState *st = nullptr;
    int rc = dev_state(&st);
    if (rc != FA_OK) return rc;
    Fp8QuantArgs a;
    a.x = x;
    a.x8 = x8;
    a.scales = scales;
    a.N = N;
    a.num_blocks = (N + 127) / 128;
    a.ld_t = a.num_blocks * 128;
    return launch_status("kernel launch",
                         launch_fp8_quant(dtype == FA_BF16, transpose != 0, a, BH, reinterpret_cast<cudaStream_t>(stream)));
}

int fa_fwd_fp8(const void *q8, const float *q_scale, const void *k8, const float *k_scale, const void *v8t,
               const float *v_scale, void *o, float *lse, int B, int H, int Nq, int Nk, int d, int causal, float scale,
               fa_dtype out_dtype, fa_stream_t stream) {
    if (q8 == nullptr || k8 == nullptr || v8t == nullptr || o == nullptr) return FA_ERR_INVALID_ARG;
    if (q_scale == nullptr || k_scale == nullptr || v_scale == nullptr) return FA_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || (long long)B * H > 65535) return FA_ERR_INVALID_ARG;
    if (!(std::isfinite(scale) && scale > 0.f) || (causal != 0 && causal != 1)) return FA_ERR_INVALID_ARG;
    if (out_dtype != FA_F16 && out_dtype != FA_BF16) return FA_ERR_INVALID_ARG;
    if (d != 128) return FA_ERR_UNSUPPORTED;
    if (!aligned(q8, 16) || !aligned(k8, 16) || !aligned(v8t, 16) || !aligned(o, 16)) return FA_ERR_MISALIGNED;
    if (!aligned(q_scale, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4)) return FA_ERR_MISALIGNED;
    if (lse != nullptr && !aligned(lse, 4)) return FA_ERR_MISALIGNED;
    DeviceState *st = nullptr;
    int rc = dev_state(&st);
    if (rc != FA_OK) return rc;
    const int BH = B * H;
    const int nbk = (Nk + 127) / 128;
    CUtensorMap tq, tk, tv;
    if ((rc = make_map_u8(&tq, q8, 128, Nq, BH)) != FA_OK || (rc = make_map_u8(&tk, k8, 128, Nk, BH)) != FA_OK ||
        (rc = make_map_u8(&tv, v8t, nbk * 128, 128, BH)) != FA_OK)
        return rc;
    Fp8FwdArgs a;
    a.o = o;
    a.lse = lse;
    a.q_scale = q_scale;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.status = st->status;
    a.Nq = Nq;
    a.Nk = Nk;
    a.num_m = (Nq + 127) / 128;
    a.causal = causal;
    a.scale_log2 = scale * 1.4426950408889634f;
    return launch_status("kernel launch", launch_fwd_fp8(out_dtype == FA_BF16, tq, tk, tv, a, BH,
                                                         reinterpret_cast<cudaStream_t>(stream)));
}

size_t fa_bwd_workspace_bytes(int B, int H, int Nq, int d) {
    if (B <= 0 || H <= 0 || Nq <= 0 || (d != 64 && d != 128)) return 0;
    const size_t rows = (size_t)B * H * (size_t)((Nq + kBwdBr - 1) / kBwdBr) * kBwdBr;
    return align256(rows * d * sizeof(float)) + 2 * align256(rows * sizeof(float));
}

int fa_bwd_gqa(const void *q, const void *k, const void *v, const void *o, const void *dout, const float *lse,
               void *dq, void *dk, void *dv, int B, int H, int H_kv, int Nq, int Nk, int d, int causal, float scale,
               fa_dtype dtype, void *workspace, size_t workspace_bytes, fa_stream_t stream) {
    int rc = check_common(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale, dtype);
    if (rc != FA_OK) return rc;
    if (H_kv <= 0 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (dout == nullptr || lse == nullptr || dq == nullptr || dk == nullptr || dv == nullptr)
        return FA_ERR_INVALID_ARG;
    if (!aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16)) return FA_ERR_MISALIGNED;
    if ((long long)B * H > 65535) return FA_ERR_INVALID_ARG;  // grid.y limit
    const size_t need = fa_bwd_workspace_bytes(B, H, Nq, d);
    if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < need) return FA_ERR_WORKSPACE;
    DeviceState *st = nullptr;
    if ((rc = dev_state(&st)) != FA_OK) return rc;
    const bool bf16 = dtype == FA_BF16;
    const int BH = B * H;
    const int Nq_pad = (Nq + kBwdBr - 1) / kBwdBr * kBwdBr;
    CUtensorMap tq, tk, tv, tdo;
    if (make_map(&tq, q, bf16, d, Nq, BH, kBwdBr) != FA_OK || make_map(&tk, k, bf16, d, Nk, B * H_kv, kBwdBc) != FA_OK ||
        make_map(&tv, v, bf16, d, Nk, B * H_kv, kBwdBc) != FA_OK || make_map(&tdo, dout, bf16, d, Nq, BH, kBwdBr) != FA_OK)
        return FA_ERR_CUDA;
    const size_t rows = (size_t)BH * Nq_pad;
    BwdArgs a{};
    a.o = o;
    a.dout = dout;
    a.lse = lse;
    a.dk = dk;
    a.dv = dv;
    a.dq = dq;
    a.dq_acc = static_cast<float *>(workspace);
    a.lse2 = reinterpret_cast<float *>(static_cast<char *>(workspace) + align256(rows * d * sizeof(float)));
    a.dvec = reinterpret_cast<float *>(reinterpret_cast<char *>(a.lse2) + align256(rows * sizeof(float)));
    a.status = st->status;
    a.BH = BH;
    a.Nq = Nq;
    a.Nk = Nk;
    a.Nq_pad = Nq_pad;
    a.H = H;
    a.group = H / H_kv;
    a.causal = causal;
    a.scale = scale;
    a.scale_log2 = scale * 1.4426950408889634f;
    cudaError_t e = launch_bwd(d, bf16, tq, tk, tv, tdo, a, reinterpret_cast<cudaStream_t>(stream));
    return launch_status("kernel launch", e);
}

// Workspace rows per head of a variable-length backward: room for every sequence
// to start on a multiple of 128 rows (sum of ceil(len / 128) * 128 over the
// sequences is at most 128 (ceil(total_q / 128) + num_seqs)).
static size_t varlen_rows_pad(int num_seqs, int total_q) {
    return (size_t)kBwdBr * ((size_t)(total_q + kBwdBr - 1) / kBwdBr + (size_t)num_seqs);
}

// Key blocks of a packed batch's backward work list: one per 128 keys of each
// sequence, at most ceil(total_k / 128) + num_seqs.
static long long bwd_varlen_capacity(int num_seqs, int total_k) {
    return (long long)(total_k + kBwdBc - 1) / kBwdBc + num_seqs;
}

size_t fa_bwd_varlen_workspace_bytes(int num_seqs, int total_q, int total_k, int H, int d) {
    if (num_seqs <= 0 || total_q <= 0 || total_k <= 0 || H <= 0 || (d != 64 && d != 128)) return 0;
    const size_t rows = (size_t)H * varlen_rows_pad(num_seqs, total_q);
    return align256((size_t)(num_seqs + 1) * sizeof(int)) + align256(rows * d * sizeof(float)) +
           2 * align256(rows * sizeof(float)) + align256(16 + 8 * (size_t)bwd_varlen_capacity(num_seqs, total_k));
}

int fa_bwd_varlen(const void *q, const void *k, const void *v, const void *o, const void *dout, const float *lse,
                  void *dq, void *dk, void *dv, const int *cu_seqlens_q, const int *cu_seqlens_k, int num_seqs,
                  int max_seqlen_k, int total_q, int total_k, int H, int H_kv, int d, int causal, float scale,
                  fa_dtype dtype, void *workspace, size_t workspace_bytes, fa_stream_t stream) {
    int rc = check_common(q, k, v, o, lse, 1, H, total_q, total_k, d, causal, scale, dtype);
    if (rc != FA_OK) return rc;
    if (dout == nullptr || lse == nullptr || dq == nullptr || dk == nullptr || dv == nullptr) return FA_ERR_INVALID_ARG;
    if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr) return FA_ERR_INVALID_ARG;
    if (!aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16)) return FA_ERR_MISALIGNED;
    if (!aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4)) return FA_ERR_MISALIGNED;
    if (num_seqs <= 0 || max_seqlen_k <= 0 || max_seqlen_k > total_k) return FA_ERR_INVALID_ARG;
    if (H_kv <= 0 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (H_kv > 65535 || bwd_varlen_capacity(num_seqs, total_k) > INT_MAX) return FA_ERR_INVALID_ARG;  // grid limits
    if ((long long)H * (long long)varlen_rows_pad(num_seqs, total_q) > INT_MAX) return FA_ERR_INVALID_ARG;
    const size_t need = fa_bwd_varlen_workspace_bytes(num_seqs, total_q, total_k, H, d);
    if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < need) return FA_ERR_WORKSPACE;
    DeviceState *st = nullptr;
    if ((rc = dev_state(&st)) != FA_OK) return rc;
    const bool bf16 = dtype == FA_BF16;
    CUtensorMap tq, tk, tv, tdo;
    if (make_map_packed(&tq, q, bf16, d, H, total_q, kBwdBr) != FA_OK ||
        make_map_packed(&tk, k, bf16, d, H_kv, total_k, kBwdBc) != FA_OK ||
        make_map_packed(&tv, v, bf16, d, H_kv, total_k, kBwdBc) != FA_OK ||
        make_map_packed(&tdo, dout, bf16, d, H, total_q, kBwdBr) != FA_OK)
        return FA_ERR_CUDA;
    const size_t rows_pad = varlen_rows_pad(num_seqs, total_q);
    const size_t rows = (size_t)H * rows_pad;
    char *ws = static_cast<char *>(workspace);
    BwdArgs a{};
    a.o = o;
    a.dout = dout;
    a.lse = lse;
    a.dk = dk;
    a.dv = dv;
    a.dq = dq;
    a.row_off = reinterpret_cast<int *>(ws);
    ws += align256((size_t)(num_seqs + 1) * sizeof(int));
    a.dq_acc = reinterpret_cast<float *>(ws);
    ws += align256(rows * d * sizeof(float));
    a.lse2 = reinterpret_cast<float *>(ws);
    ws += align256(rows * sizeof(float));
    a.dvec = reinterpret_cast<float *>(ws);
    ws += align256(rows * sizeof(float));
    int *work = reinterpret_cast<int *>(ws);  // the key-block work list
    a.status = st->status;
    a.BH = H;  // query heads per token
    a.H = H;
    a.group = H / H_kv;
    a.causal = causal;
    a.scale = scale;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    a.num_seqs = num_seqs;
    a.total_q = total_q;
    a.rows_pad = (int)rows_pad;
    cudaError_t e = launch_bwd_varlen(d, bf16, tq, tk, tv, tdo, a, work, (int)bwd_varlen_capacity(num_seqs, total_k),
                                      reinterpret_cast<cudaStream_t>(stream));
    return launch_status("kernel launch", e);
}

int fa_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout, const float *lse, void *dq,
           void *dk, void *dv, int B, int H, int Nq, int Nk, int d, int causal, float scale, fa_dtype dtype,
           void *workspace, size_t workspace_bytes, fa_stream_t stream) {
    return fa_bwd_gqa(q, k, v, o, dout, lse, dq, dk, dv, B, H, H, Nq, Nk, d, causal, scale, dtype, workspace,
                      workspace_bytes, stream);
}

int fa_get_device_status(fa_stream_t stream) {
    DeviceState *st = nullptr;
    int rc = dev_state(&st);
    if (rc != FA_OK) return rc;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
    int word = 0;
    if ((e = cudaMemcpyFromSymbol(&word, g_status_word, sizeof(int))) != cudaSuccess)
        return cuda_fail("cudaMemcpyFromSymbol", e);
    if (word != 0) {
        const int zero = 0;
        if ((e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int))) != cudaSuccess)
            return cuda_fail("cudaMemcpyToSymbol", e);
        if (word & kDevErrTimeout) return FA_ERR_DEVICE_TIMEOUT;
        if (word & kDevErrLayout) return cuda_fail("kernel", 0, "shared memory base not 1024-byte aligned");
    }
    if ((e = cudaPeekAtLastError()) != cudaSuccess) return cuda_fail("cudaPeekAtLastError", e);
    return FA_OK;
}

size_t fa_splitkv_noalloc_capacity_bytes(void) { return kNoAllocScratchBytes; }

int fa_selftest_timeout(int limit_ms, fa_stream_t stream) {
    if (limit_ms < 1 || limit_ms > 10000) return FA_ERR_INVALID_ARG;
    DeviceState *st = nullptr;
    int rc = dev_state(&st);
    if (rc != FA_OK) return rc;
    return launch_status("kernel launch", launch_selftest_timeout(st->status, limit_ms,
                                                                  reinterpret_cast<cudaStream_t>(stream)));
}

int fa_fwd_splitkv_noalloc(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int Nq,
                           int Nk, int d, int causal, float scale, fa_dtype dtype, int num_splits, fa_stream_t stream) {
    int rc = check_common(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale, dtype);
    if (rc != FA_OK) return rc;
    if (num_splits > kMaxSplits) return FA_ERR_INVALID_ARG;
    DeviceState *st = nullptr;
    if ((rc = dev_state(&st)) != FA_OK) return rc;
    const long long rows = (long long)B * H * Nq;
    if (num_splits <= 0) num_splits = auto_splits(st->num_sms, rows, Nk);
    if ((long long)num_splits * rows > INT32_MAX) return FA_ERR_INVALID_ARG;
    const size_t o_bytes = align256((size_t)num_splits * rows * d * sizeof(float));
    const size_t need = o_bytes + align256((size_t)num_splits * rows * sizeof(float));
    if (need > kNoAllocScratchBytes) return FA_ERR_SCRATCH_LIMIT;
    // The scratch array's host-side name is not a device address: look the address
    // up once per device, with that device current, and pass it to the kernels.
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cuda_fail("cudaGetDevice", cudaErrorInvalidDevice);
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_scratch_addr[dev] == nullptr) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_splitkv_scratch) != cudaSuccess || p == nullptr)
                return cuda_fail("cudaGetSymbolAddress", cudaErrorInvalidSymbol);
            g_scratch_addr[dev] = p;
        }
        scratch = g_scratch_addr[dev];
    }
    const bool bf16 = dtype == FA_BF16;
    const int BH = B * H;
    CUtensorMap tk, tv;
    if (make_map(&tk, k, bf16, d, Nk, BH, kDecBc) != FA_OK || make_map(&tv, v, bf16, d, Nk, BH, kDecBc) != FA_OK)
        return FA_ERR_CUDA;
    float *o_part = static_cast<float *>(scratch);
    float *lse_part = reinterpret_cast<float *>(static_cast<char *>(scratch) + o_bytes);
    SplitArgs a;
    a.q = q;
    a.o_part = o_part;
    a.lse_part = lse_part;
    a.status = st->status;
    a.Nq = Nq;
    a.Nk = Nk;
    a.BH = BH;
    a.H = H;
    a.group = 1;
    a.num_splits = num_splits;
    a.split_len = fa_splitkv_split_len(Nk, num_splits);
    a.causal = causal;
    a.scale_log2 = scale * 1.4426950408889634f;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = launch_splitkv(d, bf16, tk, tv, a, s);
    if (e != cudaSuccess) return cuda_fail("kernel launch", e);
    return fa_splitkv_combine(o_part, lse_part, o, lse, num_splits, B, H, Nq, d, dtype, stream);
}

}  // extern "C"
