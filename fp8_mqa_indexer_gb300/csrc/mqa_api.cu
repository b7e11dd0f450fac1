// mqa_api.cu -- the C ABI declared in include/mqa.h: argument validation, TMA
// tensor-map encoding, the paged work-schedule kernel, the optional on-device
// bounds check, the device status word, and kernel launches (the logits
// kernels and the top-k selection).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "mqa.h"
#include "launch.h"
#include "topk.h"

using namespace mqa;

// ------------------------------------------------------------ device state
// Kernel status word (bit flags from ptx.cuh).  Lives in the module's global
// memory: no allocation is made for it.
__device__ unsigned g_mqa_status;

namespace {

thread_local char t_msg[512] = "";

mqa_status fail(mqa_status s, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_msg, sizeof(t_msg), fmt, ap);
    va_end(ap);
    return s;
}

mqa_status cuda_fail(cudaError_t e, const char* what)
{
    return fail(MQA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

std::atomic<unsigned long long> g_wait_limit{4000000000ull};

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
int g_num_sms[kMaxDevices];
unsigned* g_status_ptr[kMaxDevices];

mqa_status device_state(int* dev_out, unsigned** status_out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(MQA_ERR_UNSUPPORTED, "device index %d too large", dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_status_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_mqa_status);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress(status)");
        g_status_ptr[dev] = static_cast<unsigned*>(ptr);
    }
    if (!g_num_sms[dev]) {
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
        g_num_sms[dev] = n;
    }
    *dev_out = dev;
    *status_out = g_status_ptr[dev];
    return MQA_OK;
}

// ---------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D map over a row-major [rows, cols] matrix of `esize`-byte elements with a
// [box_rows, box_cols] box; `row_bytes` (if nonzero) overrides the row stride
// (packed 4-bit elements: cols / 2 bytes).
mqa_status make_map_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize,
                       unsigned long long rows, unsigned long long cols, unsigned box_rows,
                       unsigned box_cols, CUtensorMapSwizzle swz, const char* what,
                       unsigned long long row_bytes = 0)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return fail(MQA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {row_bytes ? row_bytes : cols * (unsigned long long)esize};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(MQA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, (int)r);
    return MQA_OK;
}

// Map over a vector of n fp32 values with a box of `box` values, encoded as a
// [1, n] matrix (a second dimension of extent 1 whose stride is never used for
// addressing; it is padded to the 16-byte multiple the encoder requires).
mqa_status make_map_vec_f32(CUtensorMap* m, const void* base, unsigned long long n, unsigned box,
                            const char* what)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return fail(MQA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[2] = {n, 1};
    cuuint64_t strides[1] = {(n * 4 + 15) / 16 * 16};
    cuuint32_t boxd[2] = {box, 1};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides,
                    boxd, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(MQA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, (int)r);
    return MQA_OK;
}

// Map over [rows, cols] fp32 (or 4-byte) values whose rows start stride_bytes
// apart (a multiple of 16), with a box of one row of `cols` values.
mqa_status make_map_rows_f32(CUtensorMap* m, const void* base, unsigned long long cols,
                             unsigned long long rows, unsigned long long stride_bytes,
                             const char* what)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return fail(MQA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {stride_bytes};
    cuuint32_t boxd[2] = {(cuuint32_t)cols, 1};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides,
                    boxd, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(MQA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, (int)r);
    return MQA_OK;
}

bool aligned(const void* p, uintptr_t a)
{
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// ---------------------------------------------------------- small kernels
// Work schedules (see paged_mqa_logits_metadata and mqa_logits_metadata in
// mqa.h).  A query block b owns the 128-key tiles [lo, hi) given by Span; its
// units are numbered block by block, U in total, and SM k starts at unit
// floor(k * U / num_sms).  One CTA: each thread owns a contiguous chunk of
// blocks, a block-wide scan gives the chunk's first unit, and each thread then
// emits the schedule entries whose start unit falls inside its chunk.  With
// `check` set, entries are compared with `meta` instead of written, and a
// mismatch raises kDevErrBadSchedule.
constexpr int kMetaThreads = 1024;

struct PagedSpan {   // sequence b: tiles [0, ceil(ctx / 128))
    const int* ctx;
    __device__ int2 operator()(int b) const { return make_int2(0, paged_tiles(ctx[b])); }
};

struct DenseSpan {   // query block b: the tiles between its rows' first and last key
    Params p;
    __device__ int2 operator()(int b) const
    {
        int lo, hi;
        dense_block_tiles(p, b, lo, hi);
        return make_int2(lo, hi);
    }
};

template <class Span>
__global__ void __launch_bounds__(kMetaThreads)
    schedule_kernel(Span span, int NB, int num_sms, int* meta, int check, unsigned* status)
{
    __shared__ long long warp_tot[kMetaThreads / 32];
    // the logits kernel that follows may start its set-up now; it waits for
    // this kernel's completion before reading the schedule
    launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int chunk = (NB + kMetaThreads - 1) / kMetaThreads;
    const int c0 = min(tid * chunk, NB), c1 = min(c0 + chunk, NB);
    long long local = 0;
    for (int b = c0; b < c1; ++b) {
        const int2 t = span(b);
        local += t.y - t.x;
    }
    long long incl = local;
    for (int o = 1; o < 32; o <<= 1) {
        long long v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += v;
    }
    if (lane == 31)
        warp_tot[warp] = incl;
    __syncthreads();
    long long before = 0, U = 0;
    for (int k = 0; k < kMetaThreads / 32; ++k) {
        if (k < warp)
            before += warp_tot[k];
        U += warp_tot[k];
    }
    const long long P = before + incl - local;   // first unit of this chunk
    auto emit = [&](int k, int b, int t) {
        if (check) {
            if (meta[2 * k] != b || meta[2 * k + 1] != t)
                atomicOr(status, kDevErrBadSchedule);
        } else {
            meta[2 * k] = b;
            meta[2 * k + 1] = t;
        }
    };
    // entries whose start unit u_k = floor(k*U/num_sms) lies in [P, P + local)
    if (local > 0) {
        // smallest k with k*U >= P*num_sms
        long long k = (P * num_sms + U - 1) / U;
        int b = c0;
        long long base = P;
        int2 t = span(b);
        for (; k <= num_sms; ++k) {
            const long long u = k * U / num_sms;
            if (u >= P + local)
                break;
            while (u >= base + (t.y - t.x)) {
                base += t.y - t.x;
                ++b;
                t = span(b);
            }
            emit((int)k, b, t.x + (int)(u - base));
        }
    }
    // entries at u == U mark the end: (NB, 0)
    for (int k = tid; k <= num_sms; k += kMetaThreads) {
        const long long u = U == 0 ? 0 : (long long)k * U / num_sms;
        if (u >= U)
            emit(k, NB, 0);
    }
}

__global__ void check_dense_kernel(const int* __restrict__ ks, const int* __restrict__ ke, int S_q,
                                   int S_kv, long long ldo, int compressed, unsigned* status)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < S_q; i += gridDim.x * blockDim.x) {
        const int a = ks[i], b = ke[i];
        if (a < 0 || b > S_kv || a > b || (compressed && (long long)(b - a) > ldo))
            atomicOr(status, kDevErrBadRange);
    }
}

__global__ void check_paged_kernel(const int* __restrict__ ctx, const int* __restrict__ table, int B,
                                   int max_blocks, int block_kv, int num_blocks, unsigned* status)
{
    const long long width = (long long)max_blocks * block_kv;
    const long long total = (long long)B * max_blocks;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int b = (int)(e / max_blocks), pg = (int)(e % max_blocks);
        const int c = ctx[b];
        if (pg == 0 && (c < 0 || c > width))
            atomicOr(status, kDevErrBadContext);
        if (c > 0 && (long long)pg * block_kv < min((long long)c, width)) {
            const int id = table[e];
            if (id < 0 || id >= num_blocks)
                atomicOr(status, kDevErrBadBlock);
        }
    }
}

template <typename OutT>
__global__ void fill_rows_kernel(OutT* out, int rows, long long ldo, long long c0, long long c1)
{
    for (int r = blockIdx.x; r < rows; r += gridDim.x)
        for (long long c = c0 + threadIdx.x; c < c1; c += blockDim.x)
            out[r * ldo + c] = neg_inf<OutT>();
}

__global__ void selftest_wait_kernel(long long limit, unsigned* status)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    WaitCtx w{&abort_flag, status, limit};
    if (threadIdx.x == 0)
        wait_bounded(smem_u32(&bar), 0, w);   // nothing ever arrives
    __syncthreads();
}

mqa_status read_and_clear_status(cudaStream_t stream, unsigned* value)
{
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaStreamSynchronize");
    unsigned v = 0;
    e = cudaMemcpyFromSymbol(&v, g_mqa_status, sizeof(v));
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemcpyFromSymbol(status)");
    if (v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_mqa_status, &zero, sizeof(zero));
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaMemcpyToSymbol(status)");
    }
    *value = v;
    return MQA_OK;
}

mqa_status status_from_word(unsigned v)
{
    if (v & kDevErrTimeout)
        return fail(MQA_ERR_TIMEOUT, "a kernel wait ran out of its cycle budget");
    if (v)
        return fail(MQA_ERR_BAD_INPUT, "device bounds check failed (flags 0x%x)", v);
    return MQA_OK;
}

// Largest paged next_n: a sequence's tokens are scored in query atoms of
// kMaxN / H tokens, one launch per atom.
constexpr int kMaxNextN = 64;

int grid_for(int n)
{
    return n < 1 ? 1 : (n > 1184 ? 1184 : n);
}

}  // namespace

// ================================================================== C ABI
extern "C" {

const char* mqa_status_string(mqa_status s)
{
    switch (s) {
    case MQA_OK: return "MQA_OK";
    case MQA_ERR_INVALID_ARG: return "MQA_ERR_INVALID_ARG";
    case MQA_ERR_UNSUPPORTED: return "MQA_ERR_UNSUPPORTED";
    case MQA_ERR_CUDA: return "MQA_ERR_CUDA";
    case MQA_ERR_TIMEOUT: return "MQA_ERR_TIMEOUT";
    case MQA_ERR_BAD_INPUT: return "MQA_ERR_BAD_INPUT";
    }
    return "unknown mqa_status";
}

const char* mqa_last_error_message(void)
{
    return t_msg;
}

int mqa_get_num_sms(int device)
{
    if (device < 0 || device >= kMaxDevices)
        return -1;
    {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        if (g_num_sms[device])
            return g_num_sms[device];
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return -1;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    g_num_sms[device] = n;
    return n;
}

mqa_status mqa_set_wait_limit(unsigned long long cycles)
{
    g_wait_limit.store(cycles ? cycles : 4000000000ull);
    return MQA_OK;
}

mqa_status mqa_device_status(mqa_stream_t stream)
{
    int dev;
    unsigned* st;
    mqa_status s = device_state(&dev, &st);
    if (s != MQA_OK)
        return s;
    unsigned v = 0;
    s = read_and_clear_status((cudaStream_t)stream, &v);
    if (s != MQA_OK)
        return s;
    return status_from_word(v);
}

mqa_status mqa_selftest_wait_timeout(unsigned long long cycles, mqa_stream_t stream)
{
    int dev;
    unsigned* st;
    mqa_status s = device_state(&dev, &st);
    if (s != MQA_OK)
        return s;
    selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((long long)cycles, st);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MQA_OK : cuda_fail(e, "selftest launch");
}

mqa_status paged_mqa_logits_metadata(const int32_t* context_lens, int B, int next_n, int block_kv,
                                     int num_sms, int32_t* schedule_meta, mqa_stream_t stream)
{
    if (B < 0 || next_n < 1 || num_sms < 1)
        return fail(MQA_ERR_INVALID_ARG, "need B >= 0, next_n >= 1, num_sms >= 1");
    if (block_kv != 32 && block_kv != 64 && block_kv != 128)
        return fail(MQA_ERR_UNSUPPORTED, "block_kv must be 32, 64 or 128 (got %d)", block_kv);
    if (!schedule_meta || (B > 0 && !context_lens))
        return fail(MQA_ERR_INVALID_ARG, "null pointer");
    if (!aligned(schedule_meta, 4) || (B > 0 && !aligned(context_lens, 4)))
        return fail(MQA_ERR_INVALID_ARG, "context_lens and schedule_meta must be 4-byte aligned");
    int dev;
    unsigned* st;
    mqa_status s = device_state(&dev, &st);
    if (s != MQA_OK)
        return s;
    schedule_kernel<<<1, kMetaThreads, 0, (cudaStream_t)stream>>>(PagedSpan{context_lens}, B,
                                                                  num_sms, schedule_meta, 0, st);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MQA_OK : cuda_fail(e, "paged schedule launch");
}

namespace {
// mqa_logits and mqa_logits_scheduled: `schedule_meta` (num_sms + 1 entries
// from mqa_logits_metadata) or null for the in-kernel split.
// MX calls pass q_sf and kv_sf (UE8M0 block scales) and no kv_scale; fp4:
// MXFP4 elements (two E2M1 codes per byte, D / 2 bytes per row).  cand_mask:
// the candidate instances of the fused logits + top-k call (logits is then
// the candidate values, cand_thr the per-row thresholds or null).
mqa_status dense_call(const void* q, const void* kv, const float* kv_scale, const void* weights,
                      const int32_t* k_start, const int32_t* k_end, const int32_t* schedule_meta,
                      int sched_sms, void* logits, int S_q, int S_kv, int H, int D, int64_t ldo,
                      unsigned flags, cudaStream_t stream, const uint32_t* q_sf = nullptr,
                      const uint32_t* kv_sf = nullptr, bool fp4 = false,
                      unsigned* cand_mask = nullptr, const float* cand_thr = nullptr)
{
    const bool mx = q_sf != nullptr || kv_sf != nullptr;
    const bool compressed = (flags & MQA_COMPRESSED) != 0;
    const bool clean = (flags & MQA_CLEAN) != 0;
    const bool bf16 = (flags & MQA_OUT_BF16) != 0;
    const bool wbf16 = (flags & MQA_WEIGHTS_BF16) != 0;
    if (flags & ~(unsigned)(MQA_CLEAN | MQA_COMPRESSED | MQA_CHECK_BOUNDS | MQA_OUT_BF16 |
                            MQA_WEIGHTS_BF16))
        return fail(MQA_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags);
    if (S_q < 0 || S_kv < 0)
        return fail(MQA_ERR_INVALID_ARG, "S_q and S_kv must be >= 0");
    if (D != 64 && D != 128)
        return fail(MQA_ERR_UNSUPPORTED, "D must be 64 or 128 (got %d)", D);
    if (H != 8 && H != 32 && H != 64)
        return fail(MQA_ERR_UNSUPPORTED, "H must be 8, 32 or 64 (got %d)", H);
    if ((long long)S_q * H >= INT_MAX || S_kv > INT_MAX - 256)
        return fail(MQA_ERR_INVALID_ARG, "S_q * H or S_kv too large");
    if (!compressed && ldo < S_kv)
        return fail(MQA_ERR_INVALID_ARG, "ldo (%lld) < S_kv (%d)", (long long)ldo, S_kv);
    if (compressed && ldo < 1)
        return fail(MQA_ERR_INVALID_ARG, "compressed output needs ldo >= 1");
    if (S_q == 0)
        return MQA_OK;
    if (mx) {
        if (D != 128)
            return fail(MQA_ERR_UNSUPPORTED, "MX calls need D = 128 (four 32-element blocks)");
        if (schedule_meta)
            return fail(MQA_ERR_UNSUPPORTED, "MX calls take no schedule");
        if (!q_sf || (S_kv > 0 && !kv_sf))
            return fail(MQA_ERR_INVALID_ARG, "null pointer");
        if (!aligned(q_sf, 4) || (S_kv > 0 && !aligned(kv_sf, 16)))
            return fail(MQA_ERR_INVALID_ARG, "q_sf must be 4-byte and kv_sf 16-byte aligned");
        // the copies that spread packed E2M1 codes over shared memory read
        // from 32-byte aligned rows
        if (fp4 && (!aligned(q, 32) || (S_kv > 0 && !aligned(kv, 32))))
            return fail(MQA_ERR_INVALID_ARG, "MXFP4 q and kv must be 32-byte aligned");
    }
    if (!q || !weights || !k_start || !k_end || !logits ||
        (S_kv > 0 && (!kv || (!mx && !kv_scale))))
        return fail(MQA_ERR_INVALID_ARG, "null pointer");
    if (!aligned(q, 16) || !aligned(weights, 16) ||
        (S_kv > 0 && (!aligned(kv, 16) || (!mx && !aligned(kv_scale, 16)))))
        return fail(MQA_ERR_INVALID_ARG, "q, kv, kv_scale and weights must be 16-byte aligned");
    if (!aligned(logits, bf16 ? 2 : 4) || !aligned(k_start, 4) || !aligned(k_end, 4))
        return fail(MQA_ERR_INVALID_ARG,
                    "logits must be aligned to its element, k_start and k_end to 4 bytes");

    if (schedule_meta && (sched_sms < 1 || !aligned(schedule_meta, 4)))
        return fail(MQA_ERR_INVALID_ARG, "schedule_meta must be 4-byte aligned and num_sms >= 1");

    int dev;
    unsigned* st;
    mqa_status s = device_state(&dev, &st);
    if (s != MQA_OK)
        return s;
    const int num_sms = schedule_meta ? sched_sms : g_num_sms[dev];

    if (flags & MQA_CHECK_BOUNDS) {
        unsigned v = 0;
        s = read_and_clear_status(stream, &v);   // start from a clean word
        if (s != MQA_OK)
            return s;
        check_dense_kernel<<<grid_for((S_q + 255) / 256), 256, 0, stream>>>(
            k_start, k_end, S_q, S_kv, (long long)ldo, compressed, st);
        if (schedule_meta && S_kv > 0) {
            Params sp;
            memset(&sp, 0, sizeof(sp));
            sp.S_q = S_q;
            sp.S_kv = S_kv;
            sp.k_start = k_start;
            sp.k_end = k_end;
            sp.tok = kMaxN / H;
            schedule_kernel<<<1, kMetaThreads, 0, stream>>>(
                DenseSpan{sp}, (S_q + sp.tok - 1) / sp.tok, num_sms,
                const_cast<int32_t*>(schedule_meta), 1, st);
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return cuda_fail(e, "bounds-check launch");
        s = read_and_clear_status(stream, &v);
        if (s != MQA_OK)
            return s;
        if (v)
            return fail(MQA_ERR_BAD_INPUT, "a row range is outside [0, S_kv] or longer than ldo");
    }

    if (S_kv == 0) {
        // no keys: every row is empty; only compressed clean rows have padding
        if (compressed && clean) {
            if (bf16)
                fill_rows_kernel<<<grid_for(S_q), 256, 0, stream>>>(
                    static_cast<__nv_bfloat16*>(logits), S_q, (long long)ldo, 0, (long long)ldo);
            else
                fill_rows_kernel<<<grid_for(S_q), 256, 0, stream>>>(
                    static_cast<float*>(logits), S_q, (long long)ldo, 0, (long long)ldo);
            cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess)
                return cuda_fail(e, "fill launch");
        }
        return MQA_OK;
    }

    LaunchArgs a;
    memset(&a, 0, sizeof(a));
    // MX: 192 accumulator columns per unit (room for the scale factors in TMEM)
    const int tok = (mx ? kMxN : kMaxN) / H;
    const int N = tok * H;
    const CUtensorMapSwizzle swz = D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    // MXFP4: the copy spreads each 8 bytes of packed E2M1 codes (16 elements)
    // over 16 bytes of shared memory, so a row lands as 128 bytes laid out
    // like an E4M3 row, in the form the block-scaled MMA reads 4-bit operands
    const CUtensorMapDataType edt =
        fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const unsigned long long row_bytes = fp4 ? (unsigned long long)D / 2 : 0;
    if ((s = make_map_2d(&a.tm_q, q, edt, 1, (unsigned long long)S_q * H, D, N, D, swz, "q",
                         row_bytes)) != MQA_OK ||
        (s = make_map_2d(&a.tm_kv, kv, edt, 1, S_kv, D, kBlockKV, D, swz, "kv", row_bytes)) !=
            MQA_OK ||
        // MX: a valid map over the key scales, never used for copies
        (s = make_map_vec_f32(&a.tm_scale, mx ? (const void*)kv_sf : (const void*)kv_scale, S_kv,
                              kBlockKV, "kv_scale")) != MQA_OK ||
        (s = make_map_2d(&a.tm_w, weights,
                         wbf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                         wbf16 ? 2 : 4, S_q, H, tok, H, CU_TENSOR_MAP_SWIZZLE_NONE, "weights")) !=
            MQA_OK)
        return s;
    Params& p = a.p;
    p.logits = logits;
    p.ldo = ldo;
    p.flags = (clean ? kFlagClean : 0u) | (compressed ? kFlagCompressed : 0u);
    p.S_q = S_q;
    p.S_kv = S_kv;
    p.kv_scale = kv_scale;
    p.k_start = k_start;
    p.k_end = k_end;
    p.schedule_meta = schedule_meta;
    p.q_sf = q_sf;
    p.kv_sf = kv_sf;
    p.mx_fmt = fp4 ? kFmtE2M1 : kFmtE4M3;
    p.w_bf16 = wbf16 ? 1 : 0;
    p.cand_mask = cand_mask;
    p.cand_thr = cand_thr;
    p.width = S_kv;
    p.width_i = S_kv;
    p.tok = tok;
    p.tok0 = 0;
    p.blk_stride = tok;
    p.num_q_blocks = (S_q + tok - 1) / tok;
    p.rows = S_q;
    p.wait_limit = (long long)g_wait_limit.load();
    p.status = st;
    a.grid = num_sms;
    a.stream = stream;
    cudaError_t e = mx          ? launch_dense_mx(H, bf16, a)
                    : cand_mask ? launch_dense_cand(H, D, a)
                                : launch_dense(H, D, bf16, a);
    if (e == cudaErrorNotSupported)
        return fail(MQA_ERR_UNSUPPORTED, "no dense kernel for H=%d D=%d", H, D);
    if (e != cudaSuccess)
        return cuda_fail(e, "dense kernel launch");
    return MQA_OK;
}
}  // namespace

mqa_status mqa_logits(const void* q, const void* kv, const float* kv_scale, const void* weights,
                      const int32_t* k_start, const int32_t* k_end, void* logits, int S_q,
                      int S_kv, int H, int D, int64_t ldo, unsigned flags, mqa_stream_t stream)
{
    return dense_call(q, kv, kv_scale, weights, k_start, k_end, nullptr, 0, logits, S_q, S_kv, H,
                      D, ldo, flags, (cudaStream_t)stream);
}

mqa_status mqa_logits_scheduled(const void* q, const void* kv, const float* kv_scale,
                                const void* weights, const int32_t* k_start,
                                const int32_t* k_end, const int32_t* schedule_meta, int num_sms,
                                void* logits, int S_q, int S_kv, int H, int D, int64_t ldo,
                                unsigned flags, mqa_stream_t stream)
{
    if (!schedule_meta)
        return fail(MQA_ERR_INVALID_ARG, "null schedule_meta");
    return dense_call(q, kv, kv_scale, weights, k_start, k_end, schedule_meta, num_sms, logits,
                      S_q, S_kv, H, D, ldo, flags, (cudaStream_t)stream);
}

mqa_status mqa_logits_mx(const void* q, const uint32_t* q_sf, const void* kv, const uint32_t* kv_sf,
                         const void* weights, const int32_t* k_start, const int32_t* k_end,
                         void* logits, int S_q, int S_kv, int H, int D, int64_t ldo,
                         unsigned flags, mqa_stream_t stream)
{
    if (!q_sf || !kv_sf)
        return fail(MQA_ERR_INVALID_ARG, "null scale pointer");
    return dense_call(q, kv, nullptr, weights, k_start, k_end, nullptr, 0, logits, S_q, S_kv, H, D,
                      ldo, flags & ~(unsigned)MQA_MXFP4, (cudaStream_t)stream, q_sf, kv_sf,
                      (flags & MQA_MXFP4) != 0);
}

mqa_status mqa_logits_metadata(const int32_t* k_start, const int32_t* k_end, int S_q, int S_kv,
                               int H, int num_sms, int32_t* schedule_meta, mqa_stream_t stream)
{
    if (S_q < 0 || S_kv < 0 || num_sms < 1)
        return fail(MQA_ERR_INVALID_ARG, "need S_q >= 0, S_kv >= 0, num_sms >= 1");
    if (H != 8 && H != 32 && H != 64)
        return fail(MQA_ERR_UNSUPPORTED, "H must be 8, 32 or 64 (got %d)", H);
    if ((long long)S_q * H >= INT_MAX || S_kv > INT_MAX - 256)
        return fail(MQA_ERR_INVALID_ARG, "S_q * H or S_kv too large");
    if (!schedule_meta || (S_q > 0 && (!k_start || !k_end)))
        return fail(MQA_ERR_INVALID_ARG, "null pointer");
    if (!aligned(schedule_meta, 4) || (S_q > 0 && (!aligned(k_start, 4) || !aligned(k_end, 4))))
        return fail(MQA_ERR_INVALID_ARG, "k_start, k_end and schedule_meta must be 4-byte aligned");
    int dev;
    unsigned* st;
    mqa_status s = device_state(&dev, &st);
    if (s != MQA_OK)
        return s;
    Params sp;
    memset(&sp, 0, sizeof(sp));
    sp.S_q = S_q;
    sp.S_kv = S_kv;
    sp.k_start = k_start;
    sp.k_end = k_end;
    sp.tok = kMaxN / H;
    schedule_kernel<<<1, kMetaThreads, 0, (cudaStream_t)stream>>>(
        DenseSpan{sp}, (S_q + sp.tok - 1) / sp.tok, num_sms, schedule_meta, 0, st);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MQA_OK : cuda_fail(e, "dense schedule launch");
}

namespace {
// Host-side checks of a paged call, shared by paged_mqa_logits and
// paged_mqa_logits_noalloc (which runs them before it writes its schedule).
// Sets *nothing_to_do for B == 0.
mqa_status validate_paged(const void* q, const void* kv_cache, const void* kv_scales,
                          const void* weights, const int32_t* context_lens,
                          const int32_t* block_table, int max_blocks_per_seq,
                          const int32_t* schedule_meta, const void* logits, int B, int next_n,
                          int H, int D, int block_kv, int num_blocks, int num_sms, int64_t ldo,
                          unsigned flags, bool own_schedule, bool* nothing_to_do)
{
    // own_schedule: the call keeps the schedule itself (no schedule_meta or
    // num_sms from the caller to check)
    if (own_schedule) {
        schedule_meta = context_lens;
        num_sms = 1;
    }
    *nothing_to_do = false;
    if (flags & ~(unsigned)(MQA_CLEAN | MQA_CHECK_BOUNDS | MQA_OUT_BF16 | MQA_WEIGHTS_BF16 |
                            MQA_KV_FUSED))
        return fail((flags & MQA_COMPRESSED) ? MQA_ERR_UNSUPPORTED : MQA_ERR_INVALID_ARG,
                    "paged logits take only MQA_CLEAN, MQA_CHECK_BOUNDS, MQA_OUT_BF16, "
                    "MQA_WEIGHTS_BF16 and MQA_KV_FUSED (flags 0x%x)", flags);
    const bool fused = (flags & MQA_KV_FUSED) != 0;
    if (B < 0 || next_n < 1 || num_blocks < 1 || max_blocks_per_seq < 1 || num_sms < 1)
        return fail(MQA_ERR_INVALID_ARG,
                    "need B >= 0, next_n >= 1, num_blocks >= 1, max_blocks_per_seq >= 1, num_sms >= 1");
    if (D != 64 && D != 128)
        return fail(MQA_ERR_UNSUPPORTED, "D must be 64 or 128 (got %d)", D);
    if (H != 16 && H != 32 && H != 64)
        return fail(MQA_ERR_UNSUPPORTED, "H must be 16, 32 or 64 (got %d)", H);
    if (next_n > kMaxNextN)
        return fail(MQA_ERR_UNSUPPORTED, "next_n must be at most %d (got %d)", kMaxNextN, next_n);
    if (block_kv != 32 && block_kv != 64 && block_kv != 128)
        return fail(MQA_ERR_UNSUPPORTED, "block_kv must be 32, 64 or 128 (got %d)", block_kv);
    const long long width = (long long)max_blocks_per_seq * block_kv;
    if (ldo < width)
        return fail(MQA_ERR_INVALID_ARG, "ldo (%lld) < max_blocks_per_seq * block_kv (%lld)",
                    (long long)ldo, width);
    // fused pages: block_kv key rows then block_kv * 4 / D rows' worth of scales
    if (width > INT_MAX - 256 || (long long)num_blocks * (block_kv + 4 * block_kv / D) >= INT_MAX ||
        (long long)B * next_n * H >= INT_MAX)
        return fail(MQA_ERR_INVALID_ARG, "size too large");
    if (fused && kv_scales)
        return fail(MQA_ERR_INVALID_ARG, "kv_scales must be NULL with MQA_KV_FUSED");
    if (B == 0) {
        *nothing_to_do = true;
        return MQA_OK;
    }
    if (!q || !kv_cache || (!fused && !kv_scales) || !weights || !context_lens || !block_table ||
        !schedule_meta || !logits)
        return fail(MQA_ERR_INVALID_ARG, "null pointer");
    if (!aligned(q, 16) || !aligned(kv_cache, 16) || (!fused && !aligned(kv_scales, 16)) ||
        !aligned(weights, 16))
        return fail(MQA_ERR_INVALID_ARG,
                    "q, kv_cache, kv_scales and weights must be 16-byte aligned");
    if (!aligned(logits, (flags & MQA_OUT_BF16) ? 2 : 4) || !aligned(context_lens, 4) ||
        !aligned(block_table, 4) || !aligned(schedule_meta, 4))
        return fail(MQA_ERR_INVALID_ARG,
                    "logits must be aligned to its element, the int arrays to 4 bytes");
    return MQA_OK;
}
}  // namespace

namespace {
// paged_mqa_logits and paged_mqa_logits_mx.  MX calls pass q_sf and kv_sf
// (UE8M0 block scales, one word per query row and head, one per key slot) in
// place of kv_scales; fp4: MXFP4 elements (two E2M1 codes per byte).
mqa_status paged_call(const void* q, const void* kv_cache, const float* kv_scales,
                      const void* weights, const int32_t* context_lens, const int32_t* block_table,
                      int max_blocks_per_seq, const int32_t* schedule_meta, void* logits, int B,
                      int next_n, int H, int D, int block_kv, int num_blocks, int num_sms,
                      int64_t ldo, unsigned flags, cudaStream_t stream,
                      const uint32_t* q_sf = nullptr, const uint32_t* kv_sf = nullptr,
                      bool fp4 = false)
{
    const bool mx = kv_sf != nullptr;
    const bool fused = (flags & MQA_KV_FUSED) != 0;
    if (mx && fused)
        return fail(MQA_ERR_UNSUPPORTED, "MQA_KV_FUSED is for FP8 keys with fp32 scales");
    bool nothing = false;
    mqa_status v0 = validate_paged(q, kv_cache, mx ? (const void*)kv_sf : (const void*)kv_scales,
                                   weights, context_lens, block_table, max_blocks_per_seq,
                                   schedule_meta, logits, B, next_n, H, D, block_kv, num_blocks,
                                   num_sms, ldo, flags, false, &nothing);
    if (v0 != MQA_OK || nothing)
        return v0;
    if (mx) {
        if (D != 128)
            return fail(MQA_ERR_UNSUPPORTED, "MX calls need D = 128 (four 32-element blocks)");
        if (!q_sf || !aligned(q_sf, 4))
            return fail(MQA_ERR_INVALID_ARG, "q_sf must be non-null and 4-byte aligned");
        if (fp4 && (!aligned(q, 32) || !aligned(kv_cache, 32)))
            return fail(MQA_ERR_INVALID_ARG, "MXFP4 q and kv_cache must be 32-byte aligned");
    }
    const long long width = (long long)max_blocks_per_seq * block_kv;

    int dev;
    unsigned* st;
    mqa_status s = device_state(&dev, &st);
    if (s != MQA_OK)
        return s;

    if (flags & MQA_CHECK_BOUNDS) {
        unsigned v = 0;
        s = read_and_clear_status(stream, &v);
        if (s != MQA_OK)
            return s;
        const long long total = (long long)B * max_blocks_per_seq;
        check_paged_kernel<<<grid_for((int)min(total / 256 + 1, 100000LL)), 256, 0, stream>>>(
            context_lens, block_table, B, max_blocks_per_seq, block_kv, num_blocks, st);
        schedule_kernel<<<1, kMetaThreads, 0, stream>>>(
            PagedSpan{context_lens}, B, num_sms, const_cast<int32_t*>(schedule_meta), 1, st);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return cuda_fail(e, "bounds-check launch");
        s = read_and_clear_status(stream, &v);
        if (s != MQA_OK)
            return s;
        if (v)
            return fail(MQA_ERR_BAD_INPUT,
                        "bad paged input (flags 0x%x: 4 context length, 8 block id, 16 schedule)", v);
    }

    LaunchArgs a;
    memset(&a, 0, sizeof(a));
    const CUtensorMapSwizzle swz = D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    // MXFP4: packed E2M1 rows land as 128-byte rows (see dense_call)
    const CUtensorMapDataType edt =
        fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const unsigned long long row_bytes = fp4 ? (unsigned long long)D / 2 : 0;
    // Keys: rows of D bytes, page b's first at row b * page_rows.  Scales: a
    // [num_blocks, block_kv] map, row b at byte b * scale_stride (fused pages:
    // right after the page's keys).
    const long long page_rows = fused ? block_kv + 4LL * block_kv / D : block_kv;
    const void* scale_base = fused ? static_cast<const void*>(static_cast<const char*>(kv_cache) +
                                                              (size_t)block_kv * D)
                           : mx ? (const void*)kv_sf
                                : (const void*)kv_scales;
    const unsigned long long scale_stride =
        fused ? (unsigned long long)block_kv * (D + 4) : (unsigned long long)block_kv * 4;
    if ((s = make_map_2d(&a.tm_kv, kv_cache, edt, 1, (unsigned long long)num_blocks * page_rows, D,
                         block_kv, D, swz, "kv_cache", row_bytes)) != MQA_OK ||
        (s = make_map_rows_f32(&a.tm_scale, scale_base, block_kv, num_blocks, scale_stride,
                               "kv_scales")) != MQA_OK)
        return s;
    Params& p = a.p;
    p.logits = logits;
    p.ldo = ldo;
    p.flags = (flags & MQA_CLEAN) ? kFlagClean : 0u;
    p.context_lens = context_lens;
    p.block_table = block_table;
    p.schedule_meta = schedule_meta;
    p.B = B;
    p.next_n = next_n;
    p.block_kv = block_kv;
    p.max_blocks = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.kv_page_rows = (int)page_rows;
    p.width = width;
    p.width_i = (int)width;
    p.blk_stride = next_n;
    p.num_q_blocks = B;
    p.rows = B * next_n;
    p.w_bf16 = (flags & MQA_WEIGHTS_BF16) ? 1 : 0;
    p.q_sf = q_sf;
    p.kv_sf = kv_sf;
    p.mx_fmt = fp4 ? kFmtE2M1 : kFmtE4M3;
    p.wait_limit = (long long)g_wait_limit.load();
    p.status = st;
    a.grid = num_sms;
    a.stream = stream;
    // A sequence's next_n query tokens are split into query atoms of at most
    // kMaxN / H tokens (one accumulator of kMaxN columns holds an atom's
    // tokens x heads; kMxN for MX calls, whose scale factors share TMEM); each
    // atom is one launch over the same schedule.
    const int atom = (mx ? kMxN : kMaxN) / H;
    for (int t0 = 0; t0 < next_n; t0 += atom) {
        const int tok = next_n - t0 < atom ? next_n - t0 : atom;
        if ((s = make_map_2d(&a.tm_q, q, edt, 1, (unsigned long long)B * next_n * H, D,
                             (unsigned)(tok * H), D, swz, "q", row_bytes)) != MQA_OK ||
            (s = make_map_2d(&a.tm_w, weights,
                             (flags & MQA_WEIGHTS_BF16) ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                             (flags & MQA_WEIGHTS_BF16) ? 2 : 4, (unsigned long long)B * next_n, H,
                             (unsigned)tok, H, CU_TENSOR_MAP_SWIZZLE_NONE, "weights")) != MQA_OK)
            return s;
        p.tok = tok;
        p.tok0 = t0;
        cudaError_t e = mx ? launch_paged_mx(H, (flags & MQA_OUT_BF16) != 0, a)
                           : launch_paged(H, D, (flags & MQA_OUT_BF16) != 0, a);
        if (e == cudaErrorNotSupported)
            return fail(MQA_ERR_UNSUPPORTED, "no paged kernel for H=%d D=%d", H, D);
        if (e != cudaSuccess)
            return cuda_fail(e, "paged kernel launch");
    }
    return MQA_OK;
}
}  // namespace

mqa_status paged_mqa_logits(const void* q, const void* kv_cache, const float* kv_scales,
                            const void* weights, const int32_t* context_lens,
                            const int32_t* block_table, int max_blocks_per_seq,
                            const int32_t* schedule_meta, void* logits, int B, int next_n, int H,
                            int D, int block_kv, int num_blocks, int num_sms, int64_t ldo,
                            unsigned flags, mqa_stream_t stream)
{
    return paged_call(q, kv_cache, kv_scales, weights, context_lens, block_table,
                      max_blocks_per_seq, schedule_meta, logits, B, next_n, H, D, block_kv,
                      num_blocks, num_sms, ldo, flags, (cudaStream_t)stream);
}

mqa_status paged_mqa_logits_mx(const void* q, const uint32_t* q_sf, const void* kv_cache,
                               const uint32_t* kv_sf, const void* weights,
                               const int32_t* context_lens, const int32_t* block_table,
                               int max_blocks_per_seq, const int32_t* schedule_meta, void* logits,
                               int B, int next_n, int H, int D, int block_kv, int num_blocks,
                               int num_sms, int64_t ldo, unsigned flags, mqa_stream_t stream)
{
    if (!kv_sf || !q_sf)
        return fail(MQA_ERR_INVALID_ARG, "null scale pointer");
    return paged_call(q, kv_cache, nullptr, weights, context_lens, block_table, max_blocks_per_seq,
                      schedule_meta, logits, B, next_n, H, D, block_kv, num_blocks, num_sms, ldo,
                      flags & ~(unsigned)MQA_MXFP4, (cudaStream_t)stream, q_sf, kv_sf,
                      (flags & MQA_MXFP4) != 0);
}

// ------------------------------------------------ no-allocation paged call
// The schedule lives in this fixed array instead of a caller buffer.  In host
// code `g_noalloc_schedule` names a host-side stand-in, not a device address:
// the device address is looked up once per device with cudaGetSymbolAddress.
static __device__ __align__(256) int32_t g_noalloc_schedule[2 * (MQA_NOALLOC_MAX_SMS + 1)];

namespace {
std::mutex g_noalloc_mu;
int32_t* g_noalloc_ptr[kMaxDevices];
}  // namespace

mqa_status paged_mqa_logits_noalloc(const void* q, const void* kv_cache, const float* kv_scales,
                                    const void* weights, const int32_t* context_lens,
                                    const int32_t* block_table, int max_blocks_per_seq,
                                    void* logits, int B, int next_n, int H, int D, int block_kv,
                                    int num_blocks, int64_t ldo, unsigned flags,
                                    mqa_stream_t stream)
{
    // every host-side check runs before the first CUDA call and before the
    // shared schedule array is touched
    bool nothing = false;
    mqa_status s = validate_paged(q, kv_cache, kv_scales, weights, context_lens, block_table,
                                  max_blocks_per_seq, nullptr, logits, B, next_n, H, D, block_kv,
                                  num_blocks, 0, ldo, flags, true, &nothing);
    if (s != MQA_OK || nothing)
        return s;
    int dev;
    unsigned* st;
    s = device_state(&dev, &st);
    if (s != MQA_OK)
        return s;
    const int num_sms = g_num_sms[dev];
    if (num_sms > MQA_NOALLOC_MAX_SMS)
        return fail(MQA_ERR_UNSUPPORTED, "device has %d SMs; the fixed schedule holds at most %d",
                    num_sms, MQA_NOALLOC_MAX_SMS);
    int32_t* sched = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        if (!g_noalloc_ptr[dev]) {
            void* ptr = nullptr;
            cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_schedule);
            if (e != cudaSuccess)
                return cuda_fail(e, "cudaGetSymbolAddress(schedule)");
            g_noalloc_ptr[dev] = static_cast<int32_t*>(ptr);
        }
        sched = g_noalloc_ptr[dev];
    }
    s = paged_mqa_logits_metadata(context_lens, B, next_n, block_kv, num_sms, sched, stream);
    if (s != MQA_OK)
        return s;
    return paged_mqa_logits(q, kv_cache, kv_scales, weights, context_lens, block_table,
                            max_blocks_per_seq, sched, logits, B, next_n, H, D, block_kv,
                            num_blocks, num_sms, ldo, flags, stream);
}

// ------------------------------------------------------- top-k selection
namespace {
mqa_status launch_topk_checked(TopkParams& p, cudaStream_t stream)
{
    if (p.rows == 0)
        return MQA_OK;
    int dev;
    unsigned* st;
    mqa_status s = device_state(&dev, &st);
    if (s != MQA_OK)
        return s;
    const int cap = kTopkCtasPerSm * g_num_sms[dev];
    cudaError_t e = launch_topk(p, p.rows < cap ? p.rows : cap, stream);
    return e == cudaSuccess ? MQA_OK : cuda_fail(e, "top-k kernel launch");
}
}  // namespace

mqa_status mqa_topk_indices(const float* logits, const int32_t* k_start, const int32_t* k_end,
                            int32_t* indices, int S_q, int S_kv, int64_t ldo, int topk,
                            unsigned flags, mqa_stream_t stream)
{
    if (flags & ~(unsigned)(MQA_CLEAN | MQA_COMPRESSED))
        return fail(MQA_ERR_INVALID_ARG, "unknown or unsupported flag bits 0x%x", flags);
    const bool compressed = (flags & MQA_COMPRESSED) != 0;
    if (S_q < 0 || S_kv < 0 || topk < 1)
        return fail(MQA_ERR_INVALID_ARG, "need S_q >= 0, S_kv >= 0, topk >= 1");
    if (!compressed && ldo < S_kv)
        return fail(MQA_ERR_INVALID_ARG, "ldo (%lld) < S_kv (%d)", (long long)ldo, S_kv);
    if (compressed && ldo < 1)
        return fail(MQA_ERR_INVALID_ARG, "compressed logits need ldo >= 1");
    if (S_q == 0)
        return MQA_OK;
    if (!logits || !k_start || !k_end || !indices)
        return fail(MQA_ERR_INVALID_ARG, "null pointer");
    if (!aligned(logits, 4) || !aligned(k_start, 4) || !aligned(k_end, 4) || !aligned(indices, 4))
        return fail(MQA_ERR_INVALID_ARG, "logits, k_start, k_end, indices must be 4-byte aligned");
    TopkParams p;
    memset(&p, 0, sizeof(p));
    p.logits = logits;
    p.ldo = ldo;
    p.rows = S_q;
    p.n_cols = S_kv;
    p.k_start = k_start;
    p.k_end = k_end;
    p.compressed = compressed ? 1 : 0;
    p.topk = topk;
    p.indices = indices;
    return launch_topk_checked(p, (cudaStream_t)stream);
}

mqa_status paged_mqa_topk_indices(const float* logits, const int32_t* context_lens,
                                  int32_t* indices, int B, int next_n, int width, int64_t ldo,
                                  int topk, mqa_stream_t stream)
{
    if (B < 0 || next_n < 1 || width < 0 || topk < 1)
        return fail(MQA_ERR_INVALID_ARG, "need B >= 0, next_n >= 1, width >= 0, topk >= 1");
    if (ldo < width)
        return fail(MQA_ERR_INVALID_ARG, "ldo (%lld) < width (%d)", (long long)ldo, width);
    if ((long long)B * next_n >= INT_MAX)
        return fail(MQA_ERR_INVALID_ARG, "B * next_n too large");
    if (B == 0)
        return MQA_OK;
    if (!logits || !context_lens || !indices)
        return fail(MQA_ERR_INVALID_ARG, "null pointer");
    if (!aligned(logits, 4) || !aligned(context_lens, 4) || !aligned(indices, 4))
        return fail(MQA_ERR_INVALID_ARG, "logits, context_lens, indices must be 4-byte aligned");
    TopkParams p;
    memset(&p, 0, sizeof(p));
    p.logits = logits;
    p.ldo = ldo;
    p.rows = B * next_n;
    p.n_cols = width;
    p.context_lens = context_lens;
    p.next_n = next_n;
    p.topk = topk;
    p.indices = indices;
    return launch_topk_checked(p, (cudaStream_t)stream);
}


// ------------------------------------------------ fused logits + top-k
namespace {
struct CandLayout {
    long long ldo;   // candidate row stride (floats), a multiple of 128
    size_t vals, mask, ranges, thr, thr_f, t0, total;   // byte offsets into the workspace
};

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

CandLayout cand_layout(int S_q, int S_kv)
{
    CandLayout l;
    // a whole 128-key tile of every row fits its stride, so the candidate
    // kernel writes the mask of each line of a tile without a bounds test
    l.ldo = ((long long)(S_kv > 0 ? S_kv : 1) + 127) & ~127ll;
    const size_t rows = (size_t)(S_q > 0 ? S_q : 0);
    l.vals = 0;
    l.mask = round256(rows * (size_t)l.ldo * sizeof(float));
    // one scratch row of masks for the absent rows of a last query block
    l.ranges = l.mask + round256((rows + 1) * (size_t)(l.ldo / 32) * sizeof(unsigned));
    l.thr = l.ranges + round256(4 * rows * sizeof(int));
    l.thr_f = l.thr + round256(rows * sizeof(unsigned));
    l.t0 = l.thr_f + round256(rows * sizeof(float));
    l.total = l.t0 + round256(rows * sizeof(unsigned));
    return l;
}
}  // namespace

size_t mqa_logits_topk_workspace_size(int S_q, int S_kv)
{
    if (S_q < 0 || S_kv < 0)
        return 0;
    return cand_layout(S_q, S_kv).total;
}

mqa_status mqa_logits_topk(const void* q, const void* kv, const float* kv_scale,
                           const void* weights, const int32_t* k_start, const int32_t* k_end,
                           int32_t* indices, void* workspace, size_t workspace_bytes, int S_q,
                           int S_kv, int H, int D, int topk, unsigned flags, mqa_stream_t stream)
{
    if (flags & ~(unsigned)MQA_WEIGHTS_BF16)
        return fail(MQA_ERR_INVALID_ARG, "unknown or unsupported flag bits 0x%x", flags);
    if (S_q < 0 || S_kv < 0 || topk < 1)
        return fail(MQA_ERR_INVALID_ARG, "need S_q >= 0, S_kv >= 0, topk >= 1");
    if (D != 64 && D != 128)
        return fail(MQA_ERR_UNSUPPORTED, "D must be 64 or 128 (got %d)", D);
    if (H != 8 && H != 32 && H != 64)
        return fail(MQA_ERR_UNSUPPORTED, "H must be 8, 32 or 64 (got %d)", H);
    if ((long long)S_q * H >= INT_MAX || S_kv > INT_MAX - 256)
        return fail(MQA_ERR_INVALID_ARG, "S_q * H or S_kv too large");
    if (S_q == 0)
        return MQA_OK;
    if (!indices || !workspace || !k_start || !k_end || !q || !weights ||
        (S_kv > 0 && (!kv || !kv_scale)))
        return fail(MQA_ERR_INVALID_ARG, "null pointer");
    if (!aligned(q, 16) || !aligned(weights, 16) ||
        (S_kv > 0 && (!aligned(kv, 16) || !aligned(kv_scale, 16))))
        return fail(MQA_ERR_INVALID_ARG, "q, kv, kv_scale and weights must be 16-byte aligned");
    if (!aligned(indices, 4) || !aligned(workspace, 256) || !aligned(k_start, 4) ||
        !aligned(k_end, 4))
        return fail(MQA_ERR_INVALID_ARG,
                    "indices, k_start, k_end must be 4-byte and workspace 256-byte aligned");
    const CandLayout l = cand_layout(S_q, S_kv);
    if (workspace_bytes < l.total)
        return fail(MQA_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes,
                    l.total);
    if ((long long)S_q * l.ldo >= (1ll << 62) / 4)
        return fail(MQA_ERR_INVALID_ARG, "S_q * S_kv too large");
    int dev;
    unsigned* st;
    mqa_status s = device_state(&dev, &st);
    if (s != MQA_OK)
        return s;
    char* ws = static_cast<char*>(workspace);
    CandTopkParams cp;
    memset(&cp, 0, sizeof(cp));
    cp.k_start = k_start;
    cp.k_end = k_end;
    cp.rows = S_q;
    cp.n_cols = S_kv;
    cp.topk = topk;
    cp.ldo = l.ldo;
    cp.vals = reinterpret_cast<float*>(ws + l.vals);
    cp.mask = reinterpret_cast<unsigned*>(ws + l.mask);
    int* ranges = reinterpret_cast<int*>(ws + l.ranges);
    cp.pre_lo = ranges;
    cp.pre_hi = ranges + S_q;
    cp.rem_lo = ranges + 2 * (size_t)S_q;
    cp.rem_hi = ranges + 3 * (size_t)S_q;
    cp.thr = reinterpret_cast<unsigned*>(ws + l.thr);
    cp.thr_f = reinterpret_cast<float*>(ws + l.thr_f);
    cp.t0 = reinterpret_cast<unsigned*>(ws + l.t0);
    cp.indices = indices;
    cudaStream_t strm = (cudaStream_t)stream;
    float* vals = reinterpret_cast<float*>(ws + l.vals);
    unsigned* mask = reinterpret_cast<unsigned*>(ws + l.mask);
    const int grid = kTopkCtasPerSm * g_num_sms[dev];
    const int sel_grid = S_q < grid ? S_q : grid;
    cudaError_t e = launch_cand_split(cp, strm);
    if (e != cudaSuccess)
        return cuda_fail(e, "split kernel launch");
    // prefix: every logit, at its own column (the plain kernel, non-clean)
    s = dense_call(q, kv, kv_scale, weights, cp.pre_lo, cp.pre_hi, nullptr, 0, vals, S_q, S_kv,
                   H, D, l.ldo, flags, strm);
    if (s != MQA_OK)
        return s;
    if (S_kv > 0) {
        if ((e = launch_cand_threshold(cp, sel_grid, strm)) != cudaSuccess)
            return cuda_fail(e, "threshold kernel launch");
        // remainder: the logits at or above the prefix's topk-th largest
        s = dense_call(q, kv, kv_scale, weights, cp.rem_lo, cp.rem_hi, nullptr, 0, vals, S_q,
                       S_kv, H, D, l.ldo, flags, strm, nullptr, nullptr, false, mask, cp.thr_f);
        if (s != MQA_OK)
            return s;
    }
    if ((e = launch_cand_select(cp, sel_grid, strm)) != cudaSuccess)
        return cuda_fail(e, "select kernel launch");
    return MQA_OK;
}

}  // extern "C"
