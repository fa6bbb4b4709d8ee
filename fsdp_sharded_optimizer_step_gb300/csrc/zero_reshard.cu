// Reshard: remap every rank's shard of a per-rank array from the layout of
// one plan (N ranks) to the layout of another plan of the same units (N'
// ranks).  "ZeRO and FSDP sharding", Implementation notes: the checkpoint is
// written sharded (each rank its own shard) and resharding to a different N
// happens at load time.
//
// Target position j of rank r' in unit u holds the unit's position
// k = r' h'_u + j.  If k is a real position (k < s_u) it comes from rank
// r = k / h_u of the source layout, at Hoff_u + (k - r h_u); positions past
// s_u are padding in the target and are written as 0 (source padding is
// dropped).  One CTA per segment of the target's launch table; the element is
// copied as raw bits, so this is exact for any dtype.
#include <cuda_runtime.h>

#include <cstdint>

#include "zero_internal.h"
#include "zero_nvtx.h"

namespace {

constexpr int kThreads = 256;

struct ReshardArgs {
    const zero::Seg *to_segs;
    const zero::UnitDesc *from_units;
    const zero::UnitDesc *to_units;
    const void *src[ZERO_MAX_RANKS];  // from->n_ranks buffers of from->H elements
    void *dst[ZERO_MAX_RANKS];        // to->n_ranks buffers of to->H elements
};

// Block-cooperative copy of n elements.  When source and destination share
// their alignment inside 16 bytes, the body moves in 16-byte vectors, four
// per thread in flight; otherwise element by element.
template <typename T>
__device__ __forceinline__ void copy_run(const T *__restrict__ src, T *__restrict__ dst, int64_t n) {
    constexpr int VEC = 16 / sizeof(T);
    const int64_t sa = (reinterpret_cast<uintptr_t>(src) / sizeof(T)) % VEC;
    const int64_t da = (reinterpret_cast<uintptr_t>(dst) / sizeof(T)) % VEC;
    if (sa != da || n < 2 * VEC) {
        for (int64_t i = threadIdx.x; i < n; i += kThreads) dst[i] = src[i];
        return;
    }
    const int64_t head = (VEC - da) % VEC;
    const int64_t nvec = (n - head) / VEC;
    const uint4 *vs = reinterpret_cast<const uint4 *>(src + head);
    uint4 *vd = reinterpret_cast<uint4 *>(dst + head);
    if (threadIdx.x < head) dst[threadIdx.x] = src[threadIdx.x];
    int64_t i = threadIdx.x;
    for (; i + 3 * kThreads < nvec; i += 4 * kThreads) {
        const uint4 x0 = __ldcs(vs + i), x1 = __ldcs(vs + i + kThreads);
        const uint4 x2 = __ldcs(vs + i + 2 * kThreads), x3 = __ldcs(vs + i + 3 * kThreads);
        __stcs(vd + i, x0);
        __stcs(vd + i + kThreads, x1);
        __stcs(vd + i + 2 * kThreads, x2);
        __stcs(vd + i + 3 * kThreads, x3);
    }
    for (; i < nvec; i += kThreads) __stcs(vd + i, __ldcs(vs + i));
    for (int64_t t = head + nvec * VEC + threadIdx.x; t < n; t += kThreads) dst[t] = src[t];
}

template <typename T>
__global__ void __launch_bounds__(kThreads) k_reshard(const ReshardArgs a) {
    const zero::Seg sg = a.to_segs[blockIdx.x];
    const zero::UnitDesc fu = a.from_units[sg.unit];
    const zero::UnitDesc tu = a.to_units[sg.unit];
    T *dst = static_cast<T *>(a.dst[sg.rank]) + sg.s_off;
    const int64_t k0 = sg.g_off - tu.F;  // unit position of the segment's first element
    const int64_t k_end = k0 + sg.len;
    const int64_t real_end = k_end < fu.size ? k_end : fu.size;
    if (fu.h >= 64) {
        // the real part splits into runs that are contiguous in one source rank
        for (int64_t pos = k0; pos < real_end;) {
            const int64_t r = pos / fu.h;
            const int64_t run_end = (r + 1) * fu.h < real_end ? (r + 1) * fu.h : real_end;
            copy_run<T>(static_cast<const T *>(a.src[r]) + fu.Hoff + (pos - r * fu.h), dst + (pos - k0),
                        run_end - pos);
            pos = run_end;
        }
    } else {
        // tiny source slices: one lookup per element
        for (int64_t k = k0 + threadIdx.x; k < real_end; k += kThreads) {
            const int64_t r = static_cast<uint32_t>(k) / static_cast<uint32_t>(fu.h);
            dst[k - k0] = static_cast<const T *>(a.src[r])[fu.Hoff + (k - r * fu.h)];
        }
    }
    // target padding: zero
    const int64_t z0 = (real_end > k0 ? real_end : k0) - k0;
    for (int64_t j = z0 + threadIdx.x; j < sg.len; j += kThreads) dst[j] = T(0);
}

}  // namespace

extern "C" int zero_reshard(const zero_plan *from, const zero_plan *to, const void *const *src, void *const *dst,
                            int32_t dtype, zero_stream_t stream) {
    ZERO_NVTX_RANGE();
    if (from == nullptr || to == nullptr || src == nullptr || dst == nullptr) return ZERO_EINVAL;
    if (!from->attached || !to->attached) return ZERO_ENOTATTACHED;
    if (from->device != to->device) return ZERO_EINVAL;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { zero::set_last_cuda_error(static_cast<int>(e)); return ZERO_ECUDA; }
    if (dev != to->device) return ZERO_EINVAL;
    if (dtype != ZERO_F32 && dtype != ZERO_BF16) return ZERO_EINVAL;
    if (from->n_units != to->n_units || from->sizes != to->sizes) return ZERO_EINVAL;
    const uintptr_t esize = dtype == ZERO_F32 ? 4u : 2u;
    ReshardArgs a{};
    for (int q = 0; q < from->n_ranks; ++q) {
        if (src[q] == nullptr && from->p_pad > 0) return ZERO_EINVAL;
        if ((reinterpret_cast<uintptr_t>(src[q]) & (esize - 1)) != 0) return ZERO_EALIGN;
        a.src[q] = src[q];
    }
    for (int q = 0; q < to->n_ranks; ++q) {
        if (dst[q] == nullptr && to->p_pad > 0) return ZERO_EINVAL;
        if ((reinterpret_cast<uintptr_t>(dst[q]) & (esize - 1)) != 0) return ZERO_EALIGN;
        a.dst[q] = dst[q];
    }
    a.to_segs = to->d_segs;
    a.from_units = from->d_units;
    a.to_units = to->d_units;
    const int64_t nseg = static_cast<int64_t>(to->segs.size());
    if (nseg == 0) return ZERO_OK;
    if (nseg > 0x7FFFFFFF) return ZERO_EINVAL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == ZERO_F32) k_reshard<float><<<static_cast<unsigned>(nseg), kThreads, 0, st>>>(a);
    else k_reshard<unsigned short><<<static_cast<unsigned>(nseg), kThreads, 0, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) { zero::set_last_cuda_error(static_cast<int>(e)); return ZERO_ECUDA; }
    return ZERO_OK;
}
