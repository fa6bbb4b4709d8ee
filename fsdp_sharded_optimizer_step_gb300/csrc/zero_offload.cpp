// ZeRO-Offload: the fp32 AdamW step and its state (master, m, v) in host
// memory, updated by the host cores ("Learn: ZeRO & FSDP", section 6,
// Offloading: the optimizer states and the fp32 step go to the CPU, gradients
// go down, updated params come back; "ZeRO and FSDP sharding", Implementation
// notes: offload trades host-link bandwidth for capacity).
//
// The GPU reduce-scatters and averages the gradients (the pipelined reduce
// kernel) batch by batch; each batch's fp32 gradient shard is copied to the
// host on one copy stream; a pool of host threads updates the batch as soon
// as it has landed and writes its params to a host buffer in the full layout;
// those go back to the GPU on a second copy stream.  Copies down, host
// updates and copies up of different batches overlap.
//
// The host update performs, per element, the binary32 operations of the
// update in the order of include/zero.h, each rounded on its own: this file
// is compiled with -ffp-contract=off and without fast-math, every float
// expression is evaluated in binary32, and the update runs with the default
// floating-point environment (round to nearest even, no flush to zero) on
// every thread.  Its results equal zero_step's bit for bit.
#include <cuda_runtime.h>

#include <sched.h>

#include <atomic>
#include <cfenv>
#include <chrono>
#include <cmath>
#include <condition_variable>
#include <cstdint>
#include <cstring>
#include <functional>
#include <mutex>
#include <new>
#include <thread>
#include <vector>

#include "zero_launch.h"
#include "zero_nvtx.h"

namespace zero {
namespace {

// ------------------------------------------------------------------ worker pool
// n workers: the calling thread is worker 0, n - 1 threads wait for jobs.
class Pool {
  public:
    explicit Pool(int n) : n_(n) {
        for (int i = 1; i < n; ++i) threads_.emplace_back([this, i] { loop(i); });
    }
    ~Pool() {
        {
            std::lock_guard<std::mutex> g(mu_);
            stop_ = true;
        }
        cv_.notify_all();
        for (auto &t : threads_) t.join();
    }
    int size() const { return n_; }

    // Runs fn(worker) on every worker and returns when all have finished.
    void run(const std::function<void(int)> &fn) {
        {
            std::lock_guard<std::mutex> g(mu_);
            fn_ = &fn;
            pending_ = n_ - 1;
            ++gen_;
        }
        cv_.notify_all();
        fn(0);
        std::unique_lock<std::mutex> g(mu_);
        done_.wait(g, [this] { return pending_ == 0; });
        fn_ = nullptr;
    }

  private:
    void loop(int i) {
        uint64_t seen = 0;
        for (;;) {
            const std::function<void(int)> *fn;
            {
                std::unique_lock<std::mutex> g(mu_);
                cv_.wait(g, [&] { return stop_ || gen_ != seen; });
                if (stop_) return;
                seen = gen_;
                fn = fn_;
            }
            (*fn)(i);
            {
                std::lock_guard<std::mutex> g(mu_);
                if (--pending_ == 0) done_.notify_one();
            }
        }
    }

    int n_;
    std::vector<std::thread> threads_;
    std::mutex mu_;
    std::condition_variable cv_, done_;
    const std::function<void(int)> *fn_ = nullptr;
    int pending_ = 0;
    uint64_t gen_ = 0;
    bool stop_ = false;
};

// Runs the update with the default floating-point environment (round to
// nearest even, subnormals kept), whatever the calling thread had set.
class DefaultFpEnv {
  public:
    DefaultFpEnv() {
        fegetenv(&saved_);
        fesetenv(FE_DFL_ENV);
    }
    ~DefaultFpEnv() { fesetenv(&saved_); }

  private:
    fenv_t saved_;
};

// ------------------------------------------------------------------ the element update
// binary32 -> bfloat16, round to nearest even (add 0x7FFF plus the lowest kept
// bit, drop the low half); a NaN keeps its sign and top payload, quiet bit set.
inline uint16_t to_bf16(float x) {
    uint32_t u;
    std::memcpy(&u, &x, 4);
    const uint32_t rounded = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
    const uint32_t quiet = (u >> 16) | 0x40u;
    return static_cast<uint16_t>((u & 0x7FFFFFFFu) > 0x7F800000u ? quiet : rounded);
}

// AdamW over n consecutive shard positions ("ZeRO and FSDP sharding", Code,
// AdamW::step), in place on w, m, v; the params (PD: 0 none, 1 fp32, 2 bf16)
// to out.  SCALE: the gradient is first multiplied by the clip coefficient.
template <bool SCALE, int PD>
void update_run(const float *__restrict g, float *__restrict w, float *__restrict m, float *__restrict v,
                void *__restrict out, int64_t n, const AdamConsts c, float coef) {
    float *__restrict o32 = static_cast<float *>(out);
    uint16_t *__restrict o16 = static_cast<uint16_t *>(out);
    for (int64_t i = 0; i < n; ++i) {
        float gi = g[i];
        if (SCALE) gi = gi * coef;
        const float mi = c.b1 * m[i] + c.omb1 * gi;
        const float vi = c.b2 * v[i] + (c.omb2 * gi) * gi;
        const float den = std::sqrt(vi) / c.bc2 + c.eps;
        const float wi = w[i] * c.decay - (c.lr_bc1 * mi) / den;
        m[i] = mi;
        v[i] = vi;
        w[i] = wi;
        if (PD == 1) o32[i] = wi;
        if (PD == 2) o16[i] = to_bf16(wi);
    }
}

using UpdateFn = void (*)(const float *, float *, float *, float *, void *, int64_t, const AdamConsts, float);

UpdateFn pick_update(bool scale, int pd) {
    static const UpdateFn table[2][3] = {
        {update_run<false, 0>, update_run<false, 1>, update_run<false, 2>},
        {update_run<true, 0>, update_run<true, 1>, update_run<true, 2>},
    };
    return table[scale ? 1 : 0][pd];
}

// The clip coefficient of a finite S: min(1, max_norm / (sqrt(S) + 1e-6)) in
// binary64, rounded once to binary32 (the same operations as the device's).
float clip_coef(double S, float max_norm) {
    double c = static_cast<double>(max_norm) / (std::sqrt(S) + 1e-6);
    if (c > 1.0) c = 1.0;
    return static_cast<float>(c);
}

constexpr int64_t kPiece = 1 << 16;          // positions one worker takes at a time
constexpr int64_t kDefaultBatch = 1 << 22;   // padded elements per pipelined batch (at least)

// A contiguous run of one rank's slice of one unit.
struct Piece {
    int32_t unit, rank;
    int64_t j0, len;  // slice positions [j0, j0 + len)
};

struct Batch {
    int32_t u0, u1;         // units [u0, u1)
    int64_t p0, p1;         // pieces [p0, p1)
    int64_t F0, F1;         // full positions [F0, F1)
    int64_t H0, H1;         // shard positions [H0, H1) of every rank
};

double ms_since(std::chrono::steady_clock::time_point t0) {
    return std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
}

int cuda_fail(cudaError_t e) {
    set_last_cuda_error(static_cast<int>(e));
    return ZERO_ECUDA;
}

int usable_cores() {
    cpu_set_t set;
    if (sched_getaffinity(0, sizeof(set), &set) == 0) {
        const int n = CPU_COUNT(&set);
        if (n > 0) return n;
    }
    const unsigned n = std::thread::hardware_concurrency();
    return n > 0 ? static_cast<int>(n) : 1;
}

}  // namespace
}  // namespace zero

using namespace zero;

struct zero_offload {
    const zero_plan *plan = nullptr;
    Pool *pool = nullptr;
    std::vector<Piece> pieces;
    std::vector<int64_t> unit_piece_begin;  // [n_units + 1]
    std::vector<Batch> batches;
    // device side, made by the first step on the plan's device
    bool streams_ready = false;
    cudaStream_t d2h = nullptr, h2d = nullptr;
    cudaEvent_t ev_start = nullptr, ev_landed = nullptr, ev_sent = nullptr, ev_norm = nullptr;
    std::vector<cudaEvent_t> reduced, landed;
    // the clip's S, written by the total's kernel straight into mapped page-locked host
    // memory: a copy would queue on the copy engine behind the gradient shard's copies
    double *host_S = nullptr, *host_S_dev = nullptr;
    // timings of the last step
    double call_ms = 0, wait_ms = 0, cpu_ms = 0;
    bool stepped = false;

    ~zero_offload();
};

namespace {

// Updates pieces [p0, p1) on the engine's pool.  out_full / out_shard: the
// param outputs (full layout / shard layout, either may be null).
void update_pieces(zero_offload *eng, int64_t p0, int64_t p1, const float *const *gshard, float *const *master,
                   float *const *m, float *const *v, void *out_full, void *const *out_shard, int32_t pdtype,
                   const AdamConsts &c, bool scale, float coef) {
    if (p1 <= p0) return;
    const zero_plan *plan = eng->plan;
    const int esz = pdtype == ZERO_BF16 ? 2 : 4;
    const bool any_out = out_full != nullptr || out_shard != nullptr;
    const UpdateFn fn = pick_update(scale, any_out ? (pdtype == ZERO_BF16 ? 2 : 1) : 0);
    std::atomic<int64_t> next{p0};
    const std::function<void(int)> job = [&](int) {
        DefaultFpEnv env;
        for (int64_t k = next.fetch_add(1); k < p1; k = next.fetch_add(1)) {
            const Piece &pc = eng->pieces[k];
            const int r = pc.rank;
            const int64_t s = plan->Hoff[pc.unit] + pc.j0;                         // shard position
            const int64_t f = plan->F[pc.unit] + r * plan->h[pc.unit] + pc.j0;     // full position
            char *o1 = out_full != nullptr ? static_cast<char *>(out_full) + f * esz
                                           : (out_shard != nullptr ? static_cast<char *>(out_shard[r]) + s * esz : nullptr);
            fn(gshard[r] + s, master[r] + s, m[r] + s, v[r] + s, o1, pc.len, c, coef);
            if (out_full != nullptr && out_shard != nullptr)
                std::memcpy(static_cast<char *>(out_shard[r]) + s * esz, o1, static_cast<size_t>(pc.len) * esz);
        }
    };
    eng->pool->run(job);
}

bool host_rows_ok(const zero_plan *plan, const void *const *arr) {
    if (arr == nullptr) return false;
    for (int q = 0; q < plan->n_ranks; ++q)
        if (arr[q] == nullptr && plan->p_pad != 0) return false;
    return true;
}

int dev_rows_check(const zero_plan *plan, const void *const *arr) {
    if (arr == nullptr) return ZERO_EINVAL;
    for (int q = 0; q < plan->n_ranks; ++q) {
        if (arr[q] == nullptr) {
            if (plan->p_pad == 0) continue;
            return ZERO_EINVAL;
        }
        if ((reinterpret_cast<uintptr_t>(arr[q]) & 15u) != 0) return ZERO_EALIGN;
    }
    return ZERO_OK;
}

// Releases the copy streams, events and page-locked scalar (whatever exists).
void release_device_side(zero_offload *eng) {
    for (cudaEvent_t &ev : eng->reduced)
        if (ev != nullptr) cudaEventDestroy(ev), ev = nullptr;
    for (cudaEvent_t &ev : eng->landed)
        if (ev != nullptr) cudaEventDestroy(ev), ev = nullptr;
    for (cudaEvent_t *ev : {&eng->ev_start, &eng->ev_landed, &eng->ev_sent, &eng->ev_norm})
        if (*ev != nullptr) cudaEventDestroy(*ev), *ev = nullptr;
    for (cudaStream_t *st : {&eng->d2h, &eng->h2d})
        if (*st != nullptr) cudaStreamDestroy(*st), *st = nullptr;
    if (eng->host_S != nullptr) cudaFreeHost(eng->host_S), eng->host_S = nullptr;
    eng->host_S_dev = nullptr;
    eng->streams_ready = false;
}

// The copy streams, events and a page-locked scalar, made on the current device by
// the first step; after a failure nothing is kept and the next step tries again.
int make_device_side(zero_offload *eng) {
    if (eng->streams_ready) return ZERO_OK;
    eng->reduced.assign(eng->batches.size(), nullptr);
    eng->landed.assign(eng->batches.size(), nullptr);
    cudaError_t e = cudaStreamCreateWithFlags(&eng->d2h, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&eng->h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreate(&eng->ev_start);
    if (e == cudaSuccess) e = cudaEventCreate(&eng->ev_landed);
    if (e == cudaSuccess) e = cudaEventCreate(&eng->ev_sent);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&eng->ev_norm, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaHostAlloc(reinterpret_cast<void **>(&eng->host_S), 64, cudaHostAllocMapped);
    if (e == cudaSuccess) e = cudaHostGetDevicePointer(reinterpret_cast<void **>(&eng->host_S_dev), eng->host_S, 0);
    for (size_t b = 0; e == cudaSuccess && b < eng->batches.size(); ++b) {
        e = cudaEventCreateWithFlags(&eng->reduced[b], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&eng->landed[b], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) {
        release_device_side(eng);
        return cuda_fail(e);
    }
    eng->streams_ready = true;
    return ZERO_OK;
}

}  // namespace

zero_offload::~zero_offload() {
    release_device_side(this);
    delete pool;
}

extern "C" int zero_offload_create(const zero_plan *plan, int32_t n_threads, int64_t batch_min, zero_offload **out) {
    if (out == nullptr) return ZERO_EINVAL;
    *out = nullptr;
    if (plan == nullptr || n_threads < 0 || batch_min < 0) return ZERO_EINVAL;
    const int64_t bmin = batch_min > 0 ? batch_min : kDefaultBatch;
    zero_offload *eng = new (std::nothrow) zero_offload();
    if (eng == nullptr) return ZERO_ENOMEM;
    try {
        eng->plan = plan;
        const int U = plan->n_units, N = plan->n_ranks;
        eng->unit_piece_begin.assign(static_cast<size_t>(U) + 1, 0);
        for (int u = 0; u < U; ++u) {
            eng->unit_piece_begin[u] = static_cast<int64_t>(eng->pieces.size());
            for (int r = 0; r < N; ++r)
                for (int64_t j = 0; j < plan->h[u]; j += kPiece)
                    eng->pieces.push_back(Piece{u, r, j, std::min<int64_t>(kPiece, plan->h[u] - j)});
        }
        eng->unit_piece_begin[U] = static_cast<int64_t>(eng->pieces.size());
        // batches: consecutive units of at least bmin padded elements (the last may be smaller)
        for (int u = 0; u < U;) {
            Batch b{};
            b.u0 = u;
            int64_t elems = 0;
            while (u < U && (elems < bmin || plan->S[u] == 0)) elems += plan->S[u++];
            b.u1 = u;
            b.p0 = eng->unit_piece_begin[b.u0];
            b.p1 = eng->unit_piece_begin[b.u1];
            b.F0 = plan->F[b.u0];
            b.H0 = plan->Hoff[b.u0];
            b.F1 = b.u1 < U ? plan->F[b.u1] : plan->p_pad;
            b.H1 = b.u1 < U ? plan->Hoff[b.u1] : plan->H;
            if (b.F1 > b.F0) eng->batches.push_back(b);
        }
        const int threads = n_threads > 0 ? n_threads : usable_cores();
        eng->pool = new Pool(threads);
    } catch (...) {
        delete eng;
        return ZERO_ENOMEM;
    }
    *out = eng;
    return ZERO_OK;
}

extern "C" void zero_offload_destroy(zero_offload *eng) { delete eng; }

extern "C" int zero_offload_info(const zero_offload *eng, int32_t *n_threads, int64_t *n_batches) {
    if (eng == nullptr) return ZERO_EINVAL;
    if (n_threads != nullptr) *n_threads = eng->pool->size();
    if (n_batches != nullptr) *n_batches = static_cast<int64_t>(eng->batches.size());
    return ZERO_OK;
}

extern "C" int zero_offload_adamw(zero_offload *eng, const float *const *gshard_h, float *const *master_h,
                                  float *const *m_h, float *const *v_h, void *const *pshard_h, void *full_h,
                                  int32_t pdtype, const zero_hparams *hp, double sqnorm, int32_t unit) {
    ZERO_NVTX_RANGE();
    if (eng == nullptr || hp == nullptr) return ZERO_EINVAL;
    const zero_plan *plan = eng->plan;
    if (pdtype != ZERO_BF16 && pdtype != ZERO_F32) return ZERO_EINVAL;
    if (unit < -1 || unit >= plan->n_units) return ZERO_EINVAL;
    if (!host_rows_ok(plan, reinterpret_cast<const void *const *>(gshard_h)) ||
        !host_rows_ok(plan, reinterpret_cast<const void *const *>(master_h)) ||
        !host_rows_ok(plan, reinterpret_cast<const void *const *>(m_h)) ||
        !host_rows_ok(plan, reinterpret_cast<const void *const *>(v_h)))
        return ZERO_EINVAL;
    if (pshard_h != nullptr && !host_rows_ok(plan, pshard_h)) return ZERO_EINVAL;
    AdamConsts c;
    int rc = adam_consts(hp, &c);
    if (rc != ZERO_OK) return rc;
    float coef = 1.0f;
    const bool clip = hp->max_norm > 0.0f;
    if (clip) {
        if (!std::isfinite(sqnorm)) return ZERO_ENONFINITE;
        coef = clip_coef(sqnorm, hp->max_norm);
    }
    const int64_t p0 = unit < 0 ? 0 : eng->unit_piece_begin[unit];
    const int64_t p1 = unit < 0 ? static_cast<int64_t>(eng->pieces.size()) : eng->unit_piece_begin[unit + 1];
    try {
        update_pieces(eng, p0, p1, gshard_h, master_h, m_h, v_h, full_h, pshard_h, pdtype, c, clip, coef);
    } catch (...) {
        return ZERO_ENOMEM;
    }
    return ZERO_OK;
}

extern "C" int zero_offload_step(zero_offload *eng, const void *const *grads, int32_t gdtype,
                                 float *const *gshard_dev, float *const *gshard_h, float *const *master_h,
                                 float *const *m_h, float *const *v_h, void *full_h, void *full_dev, int32_t pdtype,
                                 const zero_hparams *hp, double *sqnorm_out, zero_stream_t stream) {
    ZERO_NVTX_RANGE();
    const auto t_call = std::chrono::steady_clock::now();
    if (eng == nullptr || hp == nullptr) return ZERO_EINVAL;
    const zero_plan *plan = eng->plan;
    if (!plan->attached) return ZERO_ENOTATTACHED;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev != plan->device) return ZERO_EINVAL;
    if ((gdtype != ZERO_BF16 && gdtype != ZERO_F32) || (pdtype != ZERO_BF16 && pdtype != ZERO_F32)) return ZERO_EINVAL;
    int rc;
    if ((rc = dev_rows_check(plan, grads)) != ZERO_OK) return rc;
    if ((rc = dev_rows_check(plan, reinterpret_cast<const void *const *>(gshard_dev))) != ZERO_OK) return rc;
    if (!host_rows_ok(plan, reinterpret_cast<const void *const *>(gshard_h)) ||
        !host_rows_ok(plan, reinterpret_cast<const void *const *>(master_h)) ||
        !host_rows_ok(plan, reinterpret_cast<const void *const *>(m_h)) ||
        !host_rows_ok(plan, reinterpret_cast<const void *const *>(v_h)) || (full_h == nullptr && plan->p_pad != 0))
        return ZERO_EINVAL;
    if (full_dev != nullptr && (reinterpret_cast<uintptr_t>(full_dev) & 15u) != 0) return ZERO_EALIGN;
    AdamConsts c;
    if ((rc = adam_consts(hp, &c)) != ZERO_OK) return rc;
    try {
        if ((rc = make_device_side(eng)) != ZERO_OK) return rc;
        const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
        const bool clip = hp->max_norm > 0.0f;
        const int N = plan->n_ranks;
        const int esz = pdtype == ZERO_BF16 ? 2 : 4;
        eng->wait_ms = eng->cpu_ms = 0.0;
        // both copy streams start after the work already queued on `stream`
        if ((e = cudaEventRecord(eng->ev_start, st)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaStreamWaitEvent(eng->d2h, eng->ev_start, 0)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaStreamWaitEvent(eng->h2d, eng->ev_start, 0)) != cudaSuccess) return cuda_fail(e);
        // 1-2: reduce each batch on the GPU, copy its gradient shard down
        for (size_t b = 0; b < eng->batches.size(); ++b) {
            const Batch &B = eng->batches[b];
            if ((rc = reduce_units(plan, B.u0, B.u1, grads, gdtype, gshard_dev, clip, st)) != ZERO_OK) return rc;
            if ((e = cudaEventRecord(eng->reduced[b], st)) != cudaSuccess) return cuda_fail(e);
            if ((e = cudaStreamWaitEvent(eng->d2h, eng->reduced[b], 0)) != cudaSuccess) return cuda_fail(e);
            const size_t bytes = static_cast<size_t>(B.H1 - B.H0) * 4;
            for (int r = 0; r < N; ++r)
                if ((e = cudaMemcpyAsync(gshard_h[r] + B.H0, gshard_dev[r] + B.H0, bytes, cudaMemcpyDeviceToHost,
                                         eng->d2h)) != cudaSuccess)
                    return cuda_fail(e);
            if ((e = cudaEventRecord(eng->landed[b], eng->d2h)) != cudaSuccess) return cuda_fail(e);
        }
        if ((e = cudaEventRecord(eng->ev_landed, eng->d2h)) != cudaSuccess) return cuda_fail(e);
        float coef = 1.0f;
        double S = 0.0;
        if (clip) {
            // the fixed-order total of every segment's sum of squares, written to the host directly
            *reinterpret_cast<volatile double *>(eng->host_S) = std::nan("");
            if ((rc = launch_finalize(plan, hp->max_norm, eng->host_S_dev, st)) != ZERO_OK) return rc;
            if ((e = cudaEventRecord(eng->ev_norm, st)) != cudaSuccess) return cuda_fail(e);
            const auto t0 = std::chrono::steady_clock::now();
            if ((e = cudaEventSynchronize(eng->ev_norm)) != cudaSuccess) return cuda_fail(e);
            eng->wait_ms += ms_since(t0);
            S = *reinterpret_cast<volatile double *>(eng->host_S);
            if (sqnorm_out != nullptr) *sqnorm_out = S;
            if (!std::isfinite(S)) {
                // skip the update: nothing of the state or the params is touched
                if ((e = cudaStreamWaitEvent(st, eng->ev_landed, 0)) != cudaSuccess) return cuda_fail(e);
                if ((e = cudaEventRecord(eng->ev_sent, eng->h2d)) != cudaSuccess) return cuda_fail(e);
                eng->stepped = true;
                eng->call_ms = ms_since(t_call);
                return ZERO_ENONFINITE;
            }
            coef = clip_coef(S, hp->max_norm);
        }
        // 3-4: update each batch on the host as it lands, copy its params up
        for (size_t b = 0; b < eng->batches.size(); ++b) {
            const Batch &B = eng->batches[b];
            auto t0 = std::chrono::steady_clock::now();
            if ((e = cudaEventSynchronize(eng->landed[b])) != cudaSuccess) return cuda_fail(e);
            eng->wait_ms += ms_since(t0);
            t0 = std::chrono::steady_clock::now();
            update_pieces(eng, B.p0, B.p1, gshard_h, master_h, m_h, v_h, full_h, nullptr, pdtype, c, clip, coef);
            eng->cpu_ms += ms_since(t0);
            if (full_dev != nullptr) {
                const size_t off = static_cast<size_t>(B.F0) * esz, bytes = static_cast<size_t>(B.F1 - B.F0) * esz;
                if ((e = cudaMemcpyAsync(static_cast<char *>(full_dev) + off, static_cast<const char *>(full_h) + off,
                                         bytes, cudaMemcpyHostToDevice, eng->h2d)) != cudaSuccess)
                    return cuda_fail(e);
            }
        }
        if ((e = cudaEventRecord(eng->ev_sent, eng->h2d)) != cudaSuccess) return cuda_fail(e);
        // later work on `stream` sees full_dev updated and may overwrite gshard_dev
        if ((e = cudaStreamWaitEvent(st, eng->ev_sent, 0)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaStreamWaitEvent(st, eng->ev_landed, 0)) != cudaSuccess) return cuda_fail(e);
    } catch (...) {
        return ZERO_ENOMEM;
    }
    eng->stepped = true;
    eng->call_ms = ms_since(t_call);
    return ZERO_OK;
}

extern "C" int zero_offload_timings(zero_offload *eng, double *ms) {
    if (eng == nullptr || ms == nullptr || !eng->stepped) return ZERO_EINVAL;
    ms[0] = eng->call_ms;
    ms[1] = eng->wait_ms;
    ms[2] = eng->cpu_ms;
    float sent = 0.f, landed = 0.f;
    cudaError_t e = cudaEventSynchronize(eng->ev_sent);
    if (e == cudaSuccess) e = cudaEventSynchronize(eng->ev_landed);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&sent, eng->ev_start, eng->ev_sent);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&landed, eng->ev_start, eng->ev_landed);
    if (e != cudaSuccess) return cuda_fail(e);
    ms[3] = sent;
    ms[4] = landed;
    return ZERO_OK;
}
