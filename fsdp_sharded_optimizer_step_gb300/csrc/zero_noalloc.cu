// zero_grad_sqnorm_noalloc: the global gradient sum of squares without any
// device allocation, for callers that cannot obtain device memory.
//
// Who needs it: a norm check that has to run exactly when memory is gone --
// logging the gradient norm while diagnosing a step that hit out-of-memory,
// or a watchdog that checks for a diverging (non-finite) gradient from inside
// a framework whose caching allocator already holds nearly all of the GPU.
// There, a cudaMalloc (or a request to the framework allocator) fails or
// forces the allocator to release and re-reserve memory, which is exactly what
// the check must not do.  This entry point needs no plan workspace and no
// caller scratch: its per-chunk partial sums live in a fixed array compiled
// into the library, which every GPU that loads the library keeps until the
// process exits.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <unordered_map>

#include "zero_internal.h"
#include "zero_nvtx.h"

namespace {

constexpr int kThreads = 256;
constexpr int64_t kChunk = ZERO_NOALLOC_CHUNK;          // elements summed by one CTA
constexpr int kMaxChunks = ZERO_NOALLOC_MAX_CHUNKS;     // capacity of the partials array

// The scratch: one binary64 partial per chunk.  Shared by every call on a
// device; a call writes partials [0, nchunks) before it reads them, so
// nothing has to start at zero, but two calls that overlap on the GPU race.
__device__ __align__(256) double g_sqnorm_scratch[kMaxChunks];

struct Args {
    const void *grads[ZERO_MAX_RANKS];
    int32_t n_ranks;
    int32_t gdtype;
    int32_t pow2;
    float inv_n, nf;
    int64_t n;
    double *partials;
};

__device__ __forceinline__ float load_one(const void *base, int32_t gdtype, int64_t i) {
    if (gdtype == ZERO_BF16) return __uint_as_float(static_cast<uint32_t>(static_cast<const unsigned short *>(base)[i]) << 16);
    return static_cast<const float *>(base)[i];
}

__device__ __forceinline__ double block_total(double x, double *smem) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = __dadd_rn(x, __shfl_down_sync(0xFFFFFFFFu, x, o));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) smem[warp] = x;
    __syncthreads();
    double s = 0.0;
    if (warp == 0) {
        s = lane < (blockDim.x >> 5) ? smem[lane] : 0.0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s = __dadd_rn(s, __shfl_down_sync(0xFFFFFFFFu, s, o));
    }
    return s;
}

// One CTA per chunk of kChunk positions: the averaged gradient (rank-ordered
// binary32 fold, divided by N) squared exactly in binary64 and added up.
__global__ void __launch_bounds__(kThreads) k_sqnorm_chunks(const Args a) {
    __shared__ double smem[kThreads / 32];
    const int64_t begin = static_cast<int64_t>(blockIdx.x) * kChunk;
    const int64_t end = begin + kChunk < a.n ? begin + kChunk : a.n;
    double sq = 0.0;
    for (int64_t i = begin + threadIdx.x; i < end; i += kThreads) {
        float acc = load_one(a.grads[0], a.gdtype, i);
        for (int q = 1; q < a.n_ranks; ++q) acc = __fadd_rn(acc, load_one(a.grads[q], a.gdtype, i));
        const float g = a.pow2 ? __fmul_rn(acc, a.inv_n) : __fdiv_rn(acc, a.nf);
        const double d = static_cast<double>(g);
        sq = __dadd_rn(sq, __dmul_rn(d, d));
    }
    const double s = block_total(sq, smem);
    if (threadIdx.x == 0) a.partials[blockIdx.x] = s;
}

// Adds the partials in a fixed order and writes the total.
__global__ void __launch_bounds__(1024) k_sqnorm_total(const double *partials, int nchunks, double *out) {
    __shared__ double smem[32];
    double s = 0.0;
    for (int i = threadIdx.x; i < nchunks; i += 1024) s = __dadd_rn(s, partials[i]);
    const double t = block_total(s, smem);
    if (threadIdx.x == 0) *out = t;
}

// Set-up, once per device, with that device current: load this file's code
// onto the device and look up the scratch array's device address.  Under
// CUDA's lazy module loading the code would otherwise be loaded at the first
// launch, and loading takes device memory: a first launch made after memory
// ran out could fail.  cudaGetSymbolAddress loads the module that holds the
// array, cudaFuncGetAttributes loads each kernel.  The address is cached per
// device ordinal, so it assumes the device's context lives as long as the
// process (a cudaDeviceReset would leave a stale address behind).
std::mutex g_lock;
std::unordered_map<int, double *> g_scratch_by_device;

int scratch_on_current_device(int dev, double **out) {
    std::lock_guard<std::mutex> guard(g_lock);
    auto it = g_scratch_by_device.find(dev);
    if (it == g_scratch_by_device.end()) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_sqnorm_scratch);
        cudaFuncAttributes attr;
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&attr, k_sqnorm_chunks);
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&attr, k_sqnorm_total);
        if (e != cudaSuccess || p == nullptr) { zero::set_last_cuda_error(static_cast<int>(e)); return ZERO_ECUDA; }
        it = g_scratch_by_device.emplace(dev, static_cast<double *>(p)).first;
    }
    *out = it->second;
    return ZERO_OK;
}

// Whether ptr is device (or managed) memory of device `dev`.  A host pointer,
// or memory of another GPU, is refused before anything is launched.
bool on_device(const void *ptr, int dev) {
    cudaPointerAttributes a;
    const cudaError_t e = cudaPointerGetAttributes(&a, ptr);
    if (e != cudaSuccess) {
        cudaGetLastError();  // reset the runtime's last-error state
        return false;
    }
    return (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) && a.device == dev;
}

}  // namespace

extern "C" int zero_grad_sqnorm_noalloc(const void *const *grads, int32_t n_ranks, int32_t gdtype, int64_t n,
                                        double *sqnorm_dev, zero_stream_t stream) {
    ZERO_NVTX_RANGE();
    if (grads == nullptr || sqnorm_dev == nullptr || n < 0) return ZERO_EINVAL;
    if (n_ranks < 1 || n_ranks > ZERO_MAX_RANKS) return ZERO_EINVAL;
    if (gdtype != ZERO_BF16 && gdtype != ZERO_F32) return ZERO_EINVAL;
    if (n > kChunk * static_cast<int64_t>(kMaxChunks)) return ZERO_ERANGE;
    if ((reinterpret_cast<uintptr_t>(sqnorm_dev) & 7u) != 0) return ZERO_EALIGN;
    const uintptr_t esize = gdtype == ZERO_BF16 ? 2u : 4u;
    Args a{};
    for (int q = 0; q < n_ranks; ++q) {
        if (n > 0 && grads[q] == nullptr) return ZERO_EINVAL;
        if ((reinterpret_cast<uintptr_t>(grads[q]) & (esize - 1)) != 0) return ZERO_EALIGN;
        a.grads[q] = grads[q];
    }
    int dev = -1;
    const cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess) { zero::set_last_cuda_error(static_cast<int>(de)); return ZERO_ECUDA; }
    double *scratch = nullptr;
    int rc = scratch_on_current_device(dev, &scratch);
    if (rc != ZERO_OK) return rc;
    if (!on_device(sqnorm_dev, dev)) return ZERO_EINVAL;
    if (n > 0)
        for (int q = 0; q < n_ranks; ++q)
            if (!on_device(grads[q], dev)) return ZERO_EINVAL;
    a.n_ranks = n_ranks;
    a.gdtype = gdtype;
    a.pow2 = (n_ranks & (n_ranks - 1)) == 0;
    a.nf = static_cast<float>(n_ranks);
    a.inv_n = a.pow2 ? 1.0f / static_cast<float>(n_ranks) : 0.0f;
    a.n = n;
    a.partials = scratch;
    const int nchunks = static_cast<int>((n + kChunk - 1) / kChunk);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (nchunks > 0) k_sqnorm_chunks<<<nchunks, kThreads, 0, st>>>(a);
    k_sqnorm_total<<<1, 1024, 0, st>>>(scratch, nchunks, sqnorm_dev);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { zero::set_last_cuda_error(static_cast<int>(e)); return ZERO_ECUDA; }
    return ZERO_OK;
}
