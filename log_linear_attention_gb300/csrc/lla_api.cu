// Host side of the C ABI declared in include/lla.h: argument validation,
// path selection (tcgen05 tensor-core path or SIMT path), workspace handling
// and the per-device error word.
#include <mutex>

#include "../../include/lla.h"
#include "lla_internal.cuh"

// One error word per device (each device holds its own copy of this variable).
__device__ int lla_device_error_word;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
int* g_err_ptr[kMaxDevices];
cudaMemPool_t g_pool[kMaxDevices];
bool g_pool_ready[kMaxDevices];

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return (dev >= 0 && dev < kMaxDevices) ? dev : -1;
}

// Device address of this device's error word (looked up once per device).
int* error_word(int dev) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, lla_device_error_word) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<int*>(p);
    }
    return g_err_ptr[dev];
}

// Library-private stream-ordered pool: freed workspace stays reserved for the
// next call instead of going back to the CUDA driver.
cudaMemPool_t workspace_pool(int dev) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_pool_ready[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return nullptr;
        uint64_t keep = UINT64_MAX;
        cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        g_pool[dev] = pool;
        g_pool_ready[dev] = true;
    }
    return g_pool[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// lla_forward_host: per device, one copy-in and one copy-out stream and the events that
// order a chunk's copies and kernels; one call at a time per device.
std::mutex g_host_mutex[kMaxDevices];
cudaStream_t g_copy_in[kMaxDevices], g_copy_out[kMaxDevices];
cudaEvent_t g_host_events[kMaxDevices][7];
bool g_host_ready[kMaxDevices];

bool host_streams_ready(int dev) {
    if (g_host_ready[dev]) return true;
    if (cudaStreamCreateWithFlags(&g_copy_in[dev], cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&g_copy_out[dev], cudaStreamNonBlocking) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    for (int i = 0; i < 7; i++) {
        if (cudaEventCreateWithFlags(&g_host_events[dev][i], cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
    }
    g_host_ready[dev] = true;
    return true;
}

struct ForwardPlan {
    bool tc;
    lla::TcPlan tcp;
    lla::SimtPlan sp;
    size_t bytes;
};

int validate_forward(const void* q, const void* k, const void* v, const float* log_a, const float* lambda,
                     const void* out, int B, int H, int T, int dk, int dv, int chunk, int dtype) {
    if (!q || !k || !v || !log_a || !lambda || !out) return LLA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_a) || !aligned16(lambda) || !aligned16(out))
        return LLA_ERR_INVALID_ARG;
    if (dtype != LLA_BF16 && dtype != LLA_F32) return LLA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || T < 1 || dk < 1 || dv < 1) return LLA_ERR_INVALID_ARG;
    if (chunk != 16 && chunk != 32 && chunk != 64 && chunk != 128) return LLA_ERR_INVALID_ARG;
    if (T % chunk != 0) return LLA_ERR_INVALID_ARG;
    if (dk > 128 || dv > 128) return LLA_ERR_UNSUPPORTED;
    if ((int64_t)B * H > 65535) return LLA_ERR_UNSUPPORTED;
    if ((int64_t)B * H * T * (dk > dv ? dk : dv) > ((int64_t)1 << 40)) return LLA_ERR_UNSUPPORTED;
    return LLA_OK;
}

bool plan_forward(int B, int H, int T, int dk, int dv, int chunk, int dtype, ForwardPlan* fp) {
    fp->tc = lla::tc_supported(dtype, dk, dv, T) && lla::make_tc_plan(B, H, T, dk, dv, &fp->tcp);
    if (fp->tc) {
        fp->bytes = fp->tcp.total_bytes;
    } else {
        if (!lla::make_simt_plan(B, H, T, dk, dv, chunk, &fp->sp)) return false;
        fp->bytes = fp->sp.total_bytes;
    }
    return true;
}

int run_forward(const ForwardPlan& fp, const void* q, const void* k, const void* v, const float* log_a,
                const float* lambda, void* out, int dtype, void* ws, int* err, cudaStream_t stream) {
    cudaError_t e = fp.tc ? lla::tc_forward(fp.tcp, q, k, v, log_a, lambda, out, ws, err, stream)
                          : lla::simt_forward(fp.sp, dtype, q, k, v, log_a, lambda, out, ws, err, stream);
    return e == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
}

}  // namespace

namespace lla {
LaunchLog*& active_launch_log() {
    static thread_local LaunchLog* log = nullptr;
    return log;
}
}  // namespace lla

extern "C" {

const char* lla_status_string(int status) {
    switch (status) {
        case LLA_OK: return "LLA_OK";
        case LLA_ERR_INVALID_ARG: return "LLA_ERR_INVALID_ARG: null, misaligned or out-of-range argument";
        case LLA_ERR_UNSUPPORTED: return "LLA_ERR_UNSUPPORTED: shape outside the kernels of this build";
        case LLA_ERR_CUDA: return "LLA_ERR_CUDA: a CUDA call or kernel launch failed";
        case LLA_ERR_TIMEOUT: return "LLA_ERR_TIMEOUT: a kernel's bounded wait ran out";
        case LLA_ERR_NOMEM: return "LLA_ERR_NOMEM: workspace missing or too small";
        case LLA_ERR_DEVICE: return "LLA_ERR_DEVICE: a kernel rejected its device-side input";
        default: return "unknown lla status";
    }
}

int lla_num_levels(int64_t T) {
    if (T <= 0) return 0;
    return lla::bitlength(T - 1) + 1;
}

size_t lla_forward_workspace_size(int B, int H, int T, int dk, int dv, int chunk, int dtype) {
    // Pointers are not inspected here; validate sizes with dummy aligned non-null pointers.
    const void* dummy = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
    if (validate_forward(dummy, dummy, dummy, static_cast<const float*>(dummy), static_cast<const float*>(dummy),
                         dummy, B, H, T, dk, dv, chunk, dtype) != LLA_OK)
        return 0;
    ForwardPlan fp;
    if (!plan_forward(B, H, T, dk, dv, chunk, dtype, &fp)) return 0;
    return fp.bytes;
}

int lla_forward_ws(const void* q, const void* k, const void* v, const float* log_a, const float* lambda, void* out,
                   int B, int H, int T, int dk, int dv, int chunk, void* stream, int dtype, void* workspace,
                   size_t workspace_bytes) {
    int st = validate_forward(q, k, v, log_a, lambda, out, B, H, T, dk, dv, chunk, dtype);
    if (st != LLA_OK) return st;
    ForwardPlan fp;
    if (!plan_forward(B, H, T, dk, dv, chunk, dtype, &fp)) return LLA_ERR_UNSUPPORTED;
    if (fp.bytes > 0 && (!workspace || workspace_bytes < fp.bytes)) return LLA_ERR_NOMEM;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return LLA_ERR_INVALID_ARG;
    const int dev = current_device();
    if (dev < 0) return LLA_ERR_CUDA;
    int* err = error_word(dev);
    if (!err) return LLA_ERR_CUDA;
    return run_forward(fp, q, k, v, log_a, lambda, out, dtype, workspace, err, static_cast<cudaStream_t>(stream));
}

int lla_forward(const void* q, const void* k, const void* v, const float* log_a, const float* lambda, void* out,
                int B, int H, int T, int dk, int dv, int chunk, void* stream, int dtype) {
    int st = validate_forward(q, k, v, log_a, lambda, out, B, H, T, dk, dv, chunk, dtype);
    if (st != LLA_OK) return st;
    ForwardPlan fp;
    if (!plan_forward(B, H, T, dk, dv, chunk, dtype, &fp)) return LLA_ERR_UNSUPPORTED;
    const int dev = current_device();
    if (dev < 0) return LLA_ERR_CUDA;
    int* err = error_word(dev);
    if (!err) return LLA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* ws = nullptr;
    if (fp.bytes > 0) {
        cudaMemPool_t pool = workspace_pool(dev);
        if (!pool) return LLA_ERR_CUDA;
        if (cudaMallocFromPoolAsync(&ws, fp.bytes, pool, s) != cudaSuccess) {
            cudaGetLastError();
            return LLA_ERR_NOMEM;
        }
    }
    st = run_forward(fp, q, k, v, log_a, lambda, out, dtype, ws, err, s);
    if (ws && cudaFreeAsync(ws, s) != cudaSuccess && st == LLA_OK) st = LLA_ERR_CUDA;
    return st;
}

int lla_forward_host(const void* q, const void* k, const void* v, const float* log_a, const float* lambda,
                     void* out, int B, int H, int T, int dk, int dv, int chunk, void* stream, int dtype) {
    int st = validate_forward(q, k, v, log_a, lambda, out, B, H, T, dk, dv, chunk, dtype);
    if (st != LLA_OK) return st;
    // the buffers must be host memory (pinned or pageable)
    for (const void* p : {q, k, v, static_cast<const void*>(log_a), static_cast<const void*>(lambda),
                          static_cast<const void*>(out)}) {
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
            cudaGetLastError();
            return LLA_ERR_INVALID_ARG;
        }
        if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return LLA_ERR_INVALID_ARG;
    }
    const int BH = B * H;
    // head groups of G consecutive (b, h) heads: [BH, T, .] rows, contiguous per group
    const int nchunks = BH < 8 ? BH : 8;
    const int G = (BH + nchunks - 1) / nchunks;
    ForwardPlan fp;
    if (!plan_forward(1, G, T, dk, dv, chunk, dtype, &fp)) return LLA_ERR_UNSUPPORTED;
    const int dev = current_device();
    if (dev < 0) return LLA_ERR_CUDA;
    int* err = error_word(dev);
    if (!err) return LLA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_host_mutex[dev]);
    if (!host_streams_ready(dev)) return LLA_ERR_CUDA;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaStream_t in_s = g_copy_in[dev], out_s = g_copy_out[dev];
    cudaMemPool_t pool = workspace_pool(dev);
    if (!pool) return LLA_ERR_CUDA;
    const size_t esz = dtype == LLA_BF16 ? 2 : 4;
    const int L = lla_num_levels(T);
    const size_t rq = (size_t)T * dk * esz, rv = (size_t)T * dv * esz, ra = (size_t)T * 4, rl = (size_t)T * L * 4;
    auto up = [](size_t x) { return (x + 1023) / 1024 * 1024; };
    const size_t slot_bytes = 2 * up(G * rq) + 2 * up(G * rv) + up(G * ra) + up(G * rl);
    char* buf = nullptr;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&buf), 2 * slot_bytes + fp.bytes, pool, cs) != cudaSuccess) {
        cudaGetLastError();
        return LLA_ERR_NOMEM;
    }
    cudaEvent_t* ev = g_host_events[dev];
    cudaError_t e = cudaEventRecord(ev[6], cs);  // the buffers exist from here on
    if (e == cudaSuccess) e = cudaStreamWaitEvent(in_s, ev[6], 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(out_s, ev[6], 0);
    char* ws = buf + 2 * slot_bytes;
    const char* hq = static_cast<const char*>(q);
    const char* hk = static_cast<const char*>(k);
    const char* hv = static_cast<const char*>(v);
    const char* ha = reinterpret_cast<const char*>(log_a);
    const char* hl = reinterpret_cast<const char*>(lambda);
    char* ho = static_cast<char*>(out);
    for (int c = 0; c < nchunks && e == cudaSuccess; c++) {
        const int h0 = c * G, g = (BH - h0) < G ? (BH - h0) : G;
        if (g <= 0) break;
        const int slot = c & 1;
        char* sb = buf + slot * slot_bytes;
        char* dq = sb;
        char* dk_ = dq + up(G * rq);
        char* dv_ = dk_ + up(G * rq);
        char* dout = dv_ + up(G * rv);
        char* da = dout + up(G * rv);
        char* dl = da + up(G * ra);
        // the slot's previous chunk has been copied out (and so computed) before it is refilled
        if (c >= 2) e = cudaStreamWaitEvent(in_s, ev[4 + slot], 0);
        auto h2d = [&](char* d, const char* h, size_t row) {
            if (e == cudaSuccess) e = cudaMemcpyAsync(d, h + (size_t)h0 * row, (size_t)g * row, cudaMemcpyHostToDevice, in_s);
        };
        h2d(dq, hq, rq);
        h2d(dk_, hk, rq);
        h2d(dv_, hv, rv);
        h2d(da, ha, ra);
        h2d(dl, hl, rl);
        if (e == cudaSuccess) e = cudaEventRecord(ev[slot], in_s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, ev[slot], 0);
        if (e != cudaSuccess) break;
        ForwardPlan fg = fp;
        if (g != G && !plan_forward(1, g, T, dk, dv, chunk, dtype, &fg)) {
            e = cudaErrorInvalidValue;
            break;
        }
        if (run_forward(fg, dq, dk_, dv_, reinterpret_cast<float*>(da), reinterpret_cast<float*>(dl), dout, dtype, ws,
                        err, cs) != LLA_OK) {
            e = cudaErrorLaunchFailure;
            break;
        }
        e = cudaEventRecord(ev[2 + slot], cs);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(out_s, ev[2 + slot], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(ho + (size_t)h0 * rv, dout, (size_t)g * rv, cudaMemcpyDeviceToHost, out_s);
        if (e == cudaSuccess) e = cudaEventRecord(ev[4 + slot], out_s);
    }
    // everything has landed in host memory before the buffers go back to the pool
    const cudaError_t s1 = cudaStreamSynchronize(out_s);
    const cudaError_t s2 = cudaStreamSynchronize(in_s);
    const cudaError_t f = cudaFreeAsync(buf, cs);
    const cudaError_t s3 = cudaStreamSynchronize(cs);
    if (e != cudaSuccess || s1 != cudaSuccess || s2 != cudaSuccess || f != cudaSuccess || s3 != cudaSuccess) {
        cudaGetLastError();
        return LLA_ERR_CUDA;
    }
    return LLA_OK;
}

}  // extern "C"

namespace {

// Runs `call` (which enqueues one library call on `stream`) with the launch log active:
// a CUDA event before the first kernel and after each launch; writes each kernel's device
// time (ms) and name, in launch order, for i < cap. Returns the number of kernels launched
// or a negative lla_status.
template <typename Fn>
int profile_call(cudaStream_t s, float* kernel_ms, const char** kernel_names, int cap, Fn call) {
    if (cap < 0 || (cap > 0 && (!kernel_ms || !kernel_names))) return LLA_ERR_INVALID_ARG;
    lla::LaunchLog log;
    log.count = 0;
    cudaEvent_t start;
    if (cudaEventCreate(&start) != cudaSuccess) return LLA_ERR_CUDA;
    int made = 0;
    for (; made < lla::LaunchLog::kMax; made++)
        if (cudaEventCreate(&log.events[made]) != cudaSuccess) break;
    if (made < lla::LaunchLog::kMax) {
        for (int i = 0; i < made; i++) cudaEventDestroy(log.events[i]);
        cudaEventDestroy(start);
        return LLA_ERR_CUDA;
    }
    cudaEventRecord(start, s);
    lla::active_launch_log() = &log;
    int st = call();
    lla::active_launch_log() = nullptr;
    int n = log.count < lla::LaunchLog::kMax ? log.count : lla::LaunchLog::kMax;
    if (st == LLA_OK && n > 0 && cudaEventSynchronize(log.events[n - 1]) != cudaSuccess) st = LLA_ERR_CUDA;
    if (st == LLA_OK) {
        cudaEvent_t prev = start;
        for (int i = 0; i < n && i < cap; i++) {
            float ms = 0.f;
            cudaEventElapsedTime(&ms, prev, log.events[i]);
            kernel_ms[i] = ms;
            kernel_names[i] = log.names[i];
            prev = log.events[i];
        }
    }
    for (int i = 0; i < lla::LaunchLog::kMax; i++) cudaEventDestroy(log.events[i]);
    cudaEventDestroy(start);
    return st == LLA_OK ? log.count : st;
}

}  // namespace

extern "C" {

int lla_forward_profile(const void* q, const void* k, const void* v, const float* log_a, const float* lambda,
                        void* out, int B, int H, int T, int dk, int dv, int chunk, void* stream, int dtype,
                        float* kernel_ms, const char** kernel_names, int cap) {
    int st = validate_forward(q, k, v, log_a, lambda, out, B, H, T, dk, dv, chunk, dtype);
    if (st != LLA_OK) return st;
    return profile_call(static_cast<cudaStream_t>(stream), kernel_ms, kernel_names, cap, [&] {
        return lla_forward(q, k, v, log_a, lambda, out, B, H, T, dk, dv, chunk, stream, dtype);
    });
}

int lla_gdn_forward_profile(const void* q, const void* k, const void* v, const float* log_a, const float* beta,
                            const float* lambda, void* out, int B, int H, int T, int dk, int dv, int chunk,
                            void* stream, int dtype, float* kernel_ms, const char** kernel_names, int cap) {
    int st = validate_forward(q, k, v, log_a, lambda, out, B, H, T, dk, dv, chunk, dtype);
    if (st != LLA_OK) return st;
    return profile_call(static_cast<cudaStream_t>(stream), kernel_ms, kernel_names, cap, [&] {
        return lla_gdn_forward(q, k, v, log_a, beta, lambda, out, B, H, T, dk, dv, chunk, stream, dtype);
    });
}

int lla_decode_step(const void* q, const void* k, const void* v, const float* log_a, const float* lambda,
                    float* fenwick_states, const int64_t* t, void* out, void* stream, int B, int H, int dk, int dv,
                    int Lmax, int dtype) {
    if (!q || !k || !v || !log_a || !lambda || !fenwick_states || !t || !out) return LLA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_a) || !aligned16(lambda) ||
        !aligned16(fenwick_states) || !aligned16(t) || !aligned16(out))
        return LLA_ERR_INVALID_ARG;
    if (dtype != LLA_BF16 && dtype != LLA_F32) return LLA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || dk < 1 || dv < 1 || Lmax < 1 || Lmax > 40) return LLA_ERR_INVALID_ARG;
    if (dk > 256 || (dv != 16 && dv != 32 && dv != 64 && dv != 128)) return LLA_ERR_UNSUPPORTED;
    if ((int64_t)B * H > 0x7fffffff) return LLA_ERR_UNSUPPORTED;
    const int dev = current_device();
    if (dev < 0) return LLA_ERR_CUDA;
    int* err = error_word(dev);
    if (!err) return LLA_ERR_CUDA;
    cudaError_t e = lla::decode_step(dtype, q, k, v, log_a, lambda, fenwick_states, t, out, B, H, dk, dv, Lmax, err,
                                     static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
}

int lla_prefill_state(const void* k, const void* v, const float* log_a, float* fenwick_states, int B, int H, int T,
                      int dk, int dv, int Lmax, void* stream, int dtype) {
    if (!k || !v || !log_a || !fenwick_states) return LLA_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(log_a) || !aligned16(fenwick_states)) return LLA_ERR_INVALID_ARG;
    if (dtype != LLA_BF16 && dtype != LLA_F32) return LLA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || T < 1 || dk < 1 || dv < 1 || Lmax < 1 || Lmax > 40) return LLA_ERR_INVALID_ARG;
    if (lla::bitlength((int64_t)T - 1) + 1 > Lmax) return LLA_ERR_INVALID_ARG;
    if (dk > 128 || dv > 128) return LLA_ERR_UNSUPPORTED;
    if ((int64_t)B * H > 65535 || (int64_t)B * H * T * (dk > dv ? dk : dv) > ((int64_t)1 << 40)) return LLA_ERR_UNSUPPORTED;
    const int dev = current_device();
    if (dev < 0) return LLA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool tc = lla::tc_state_supported(dtype, dk, dv, B, H, T);
    const size_t bytes = tc ? lla::tc_state_workspace_bytes(B, H, T, dv) : (size_t)B * H * T * sizeof(float);
    int* err = error_word(dev);
    if (!err) return LLA_ERR_CUDA;
    cudaMemPool_t pool = workspace_pool(dev);
    if (!pool) return LLA_ERR_CUDA;
    void* ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, bytes, pool, s) != cudaSuccess) {
        cudaGetLastError();
        return LLA_ERR_NOMEM;
    }
    cudaError_t e = tc ? lla::tc_prefill_state(k, v, log_a, fenwick_states, B, H, T, dv, Lmax, ws, err, s)
                       : lla::prefill_state(dtype, k, v, log_a, fenwick_states, B, H, T, dk, dv, Lmax, ws, err, s);
    const cudaError_t f = cudaFreeAsync(ws, s);
    return (e == cudaSuccess && f == cudaSuccess) ? LLA_OK : LLA_ERR_CUDA;
}

int lla_backward(const void* q, const void* k, const void* v, const float* log_a, const float* lambda,
                 const void* dout, void* dq, void* dk, void* dv, float* dlog_a, float* dlambda, int B, int H, int T,
                 int dk_, int dv_, int chunk, void* stream, int dtype) {
    int st = validate_forward(q, k, v, log_a, lambda, dout, B, H, T, dk_, dv_, chunk, dtype);
    if (st != LLA_OK) return st;
    if (!dq || !dk || !dv || !dlog_a || !dlambda) return LLA_ERR_INVALID_ARG;
    if (!aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(dlog_a) || !aligned16(dlambda))
        return LLA_ERR_INVALID_ARG;
    lla::TcPlan tp;
    lla::BwdPlan bp;
    const bool tc = lla::tc_bwd_supported(dtype, dk_, dv_, T) && lla::make_tc_plan(B, H, T, dk_, dv_, &tp);
    if (!tc && !lla::make_bwd_plan(B, H, T, dk_, dv_, chunk, &bp)) return LLA_ERR_UNSUPPORTED;
    const int dev = current_device();
    if (dev < 0) return LLA_ERR_CUDA;
    int* err = error_word(dev);
    if (!err) return LLA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaMemPool_t pool = workspace_pool(dev);
    if (!pool) return LLA_ERR_CUDA;
    void* ws = nullptr;
    const size_t bytes = tc ? lla::tc_bwd_workspace_bytes(tp) : bp.total_bytes;
    if (cudaMallocFromPoolAsync(&ws, bytes, pool, s) != cudaSuccess) {
        cudaGetLastError();
        return LLA_ERR_NOMEM;
    }
    cudaError_t e = tc ? lla::tc_backward(tp, q, k, v, log_a, lambda, dout, dq, dk, dv, dlog_a, dlambda, ws, err, s)
                       : lla::simt_backward(bp, dtype, q, k, v, log_a, lambda, dout, dq, dk, dv, dlog_a, dlambda, ws,
                                            s);
    const cudaError_t f = cudaFreeAsync(ws, s);
    return (e == cudaSuccess && f == cudaSuccess) ? LLA_OK : LLA_ERR_CUDA;
}

int lla_forward_varlen(const void* q, const void* k, const void* v, const float* log_a, const float* lambda,
                       void* out, const int32_t* cu_seqlens, int n_seq, int H, int total_T, int max_T, int dk, int dv,
                       int chunk, void* stream, int dtype) {
    if (!cu_seqlens || !aligned16(cu_seqlens)) return LLA_ERR_INVALID_ARG;
    if (n_seq < 1 || max_T < 1 || total_T < 1) return LLA_ERR_INVALID_ARG;
    if ((int64_t)n_seq * max_T < total_T) return LLA_ERR_INVALID_ARG;
    const int Tpad = (max_T + 127) / 128 * 128;
    int st = validate_forward(q, k, v, log_a, lambda, out, n_seq, H, Tpad, dk, dv, chunk, dtype);
    if (st != LLA_OK) return st;
    if ((int64_t)H * total_T * (dk > dv ? dk : dv) > ((int64_t)1 << 40)) return LLA_ERR_UNSUPPORTED;
    const int dev = current_device();
    if (dev < 0) return LLA_ERR_CUDA;
    int* err = error_word(dev);
    if (!err) return LLA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaMemPool_t pool = workspace_pool(dev);
    if (!pool) return LLA_ERR_CUDA;
    const int L_in = lla_num_levels(max_T), L_pad = lla_num_levels(Tpad);
    lla::TcPlan tp;
    if (lla::tc_varlen_supported(dtype, dk, dv) && (int64_t)H * total_T < ((int64_t)1 << 31) &&
        lla::make_tc_plan(n_seq, H, Tpad, dk, dv, &tp)) {
        // tensor-core kernels over each sequence's own tiles of the packed layout: no padding
        const size_t tbytes = lla::tc_varlen_table_bytes(n_seq);
        char* ws = nullptr;
        if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&ws), tp.total_bytes + tbytes, pool, s) != cudaSuccess) {
            cudaGetLastError();
            return LLA_ERR_NOMEM;
        }
        const cudaError_t e = lla::tc_forward_varlen(tp, q, k, v, log_a, lambda, out, cu_seqlens, total_T, max_T,
                                                     L_in, ws, ws + tp.total_bytes, err, s);
        const cudaError_t f = cudaFreeAsync(ws, s);
        return (e == cudaSuccess && f == cudaSuccess) ? LLA_OK : LLA_ERR_CUDA;
    }
    ForwardPlan fp;
    if (!plan_forward(n_seq, H, Tpad, dk, dv, chunk, dtype, &fp)) return LLA_ERR_UNSUPPORTED;
    const int esz = dtype == LLA_BF16 ? 2 : 4;
    const size_t rows = (size_t)n_seq * H * Tpad;
    auto up = [](size_t x) { return (x + 1023) / 1024 * 1024; };
    const size_t bq = up(rows * dk * esz), bv = up(rows * dv * esz), ba = up(rows * 4), bl = up(rows * L_pad * 4);
    const size_t bytes = 2 * bq + 2 * bv + ba + bl + fp.bytes;
    char* ws = nullptr;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&ws), bytes, pool, s) != cudaSuccess) {
        cudaGetLastError();
        return LLA_ERR_NOMEM;
    }
    char* pq = ws;
    char* pk = pq + bq;
    char* pv = pk + bq;
    char* po = pv + bv;
    float* pa = reinterpret_cast<float*>(po + bv);
    float* pl = reinterpret_cast<float*>(po + bv + ba);
    char* fws = po + bv + ba + bl;
    cudaError_t e = cudaSuccess;
    auto chain = [&](cudaError_t x) {
        if (e == cudaSuccess) e = x;
    };
    chain(lla::varlen_pack(esz, q, pq, cu_seqlens, n_seq, H, total_T, Tpad, dk, dk, max_T, err, s));
    chain(lla::varlen_pack(esz, k, pk, cu_seqlens, n_seq, H, total_T, Tpad, dk, dk, max_T, err, s));
    chain(lla::varlen_pack(esz, v, pv, cu_seqlens, n_seq, H, total_T, Tpad, dv, dv, max_T, err, s));
    chain(lla::varlen_pack(4, log_a, pa, cu_seqlens, n_seq, H, total_T, Tpad, 1, 1, max_T, err, s));
    chain(lla::varlen_pack(4, lambda, pl, cu_seqlens, n_seq, H, total_T, Tpad, L_in, L_pad, max_T, err, s));
    if (e == cudaSuccess && run_forward(fp, pq, pk, pv, pa, pl, po, dtype, fws, err, s) != LLA_OK) e = cudaErrorUnknown;
    chain(lla::varlen_unpack(esz, po, out, cu_seqlens, n_seq, H, total_T, Tpad, dv, max_T, err, s));
    const cudaError_t f = cudaFreeAsync(ws, s);
    return (e == cudaSuccess && f == cudaSuccess) ? LLA_OK : LLA_ERR_CUDA;
}

int lla_prefill_state_varlen(const void* k, const void* v, const float* log_a, const int32_t* cu_seqlens,
                             float* fenwick_states, int n_seq, int H, int total_T, int max_T, int dk, int dv, int Lmax,
                             void* stream, int dtype) {
    if (!k || !v || !log_a || !cu_seqlens || !fenwick_states) return LLA_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(log_a) || !aligned16(cu_seqlens) || !aligned16(fenwick_states))
        return LLA_ERR_INVALID_ARG;
    if (dtype != LLA_BF16 && dtype != LLA_F32) return LLA_ERR_INVALID_ARG;
    if (n_seq < 1 || H < 1 || total_T < 1 || max_T < 1 || dk < 1 || dv < 1 || Lmax < 1 || Lmax > 40)
        return LLA_ERR_INVALID_ARG;
    if ((int64_t)n_seq * max_T < total_T) return LLA_ERR_INVALID_ARG;
    if (lla::bitlength((int64_t)max_T - 1) + 1 > Lmax) return LLA_ERR_INVALID_ARG;
    if (dk > 128 || dv > 128) return LLA_ERR_UNSUPPORTED;
    if ((int64_t)n_seq * H > 65535 || (int64_t)H * total_T * (dk > dv ? dk : dv) > ((int64_t)1 << 40))
        return LLA_ERR_UNSUPPORTED;
    const int dev = current_device();
    if (dev < 0) return LLA_ERR_CUDA;
    int* err = error_word(dev);
    if (!err) return LLA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaMemPool_t pool = workspace_pool(dev);
    if (!pool) return LLA_ERR_CUDA;
    const bool tc = lla::tc_state_supported_packed(dtype, dk, dv, n_seq, H, total_T, max_T);
    const size_t bytes = tc ? lla::tc_state_workspace_bytes(n_seq, H, max_T, dv) : (size_t)H * total_T * sizeof(float);
    void* ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, bytes, pool, s) != cudaSuccess) {
        cudaGetLastError();
        return LLA_ERR_NOMEM;
    }
    cudaError_t e = tc ? lla::tc_prefill_state(k, v, log_a, fenwick_states, n_seq, H, max_T, dv, Lmax, ws, err, s,
                                               cu_seqlens, total_T)
                       : lla::prefill_state(dtype, k, v, log_a, fenwick_states, n_seq, H, max_T, dk, dv, Lmax, ws,
                                            err, s, cu_seqlens, total_T);
    const cudaError_t f = cudaFreeAsync(ws, s);
    return (e == cudaSuccess && f == cudaSuccess) ? LLA_OK : LLA_ERR_CUDA;
}

int lla_gdn_forward(const void* q, const void* k, const void* v, const float* log_a, const float* beta,
                    const float* lambda, void* out, int B, int H, int T, int dk, int dv, int chunk, void* stream,
                    int dtype) {
    int st = validate_forward(q, k, v, log_a, lambda, out, B, H, T, dk, dv, chunk, dtype);
    if (st != LLA_OK) return st;
    if (!beta || !aligned16(beta)) return LLA_ERR_INVALID_ARG;
    lla::GdnPlan pl;
    if (dv % 16 != 0 || !lla::make_gdn_plan(B, H, T, dk, dv, chunk, &pl)) return LLA_ERR_UNSUPPORTED;
    const int dev = current_device();
    if (dev < 0) return LLA_ERR_CUDA;
    int* err = error_word(dev);
    if (!err) return LLA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaMemPool_t pool = workspace_pool(dev);
    if (!pool) return LLA_ERR_CUDA;
    void* ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, pl.total_bytes, pool, s) != cudaSuccess) {
        cudaGetLastError();
        return LLA_ERR_NOMEM;
    }
    const cudaError_t e = lla::gdn_forward(pl, dtype, q, k, v, log_a, beta, lambda, out, ws, err, s);
    const cudaError_t f = cudaFreeAsync(ws, s);
    return (e == cudaSuccess && f == cudaSuccess) ? LLA_OK : LLA_ERR_CUDA;
}

int lla_gdn_decode_step(const void* q, const void* k, const void* v, const float* log_a, const float* beta,
                        const float* lambda, float* fenwick_states, const int64_t* t, void* out, void* stream, int B,
                        int H, int dk, int dv, int Lmax, int dtype) {
    if (!q || !k || !v || !log_a || !beta || !lambda || !fenwick_states || !t || !out) return LLA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_a) || !aligned16(beta) ||
        !aligned16(lambda) || !aligned16(fenwick_states) || !aligned16(t) || !aligned16(out))
        return LLA_ERR_INVALID_ARG;
    if (dtype != LLA_BF16 && dtype != LLA_F32) return LLA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || dk < 1 || dv < 1 || Lmax < 1 || Lmax > 40) return LLA_ERR_INVALID_ARG;
    if ((dk != 16 && dk != 32 && dk != 64 && dk != 128) || (dv != 16 && dv != 32 && dv != 64 && dv != 128))
        return LLA_ERR_UNSUPPORTED;
    if ((int64_t)B * H > 0x7fffffff) return LLA_ERR_UNSUPPORTED;
    const int dev = current_device();
    if (dev < 0) return LLA_ERR_CUDA;
    int* err = error_word(dev);
    if (!err) return LLA_ERR_CUDA;
    cudaError_t e = lla::gdn_decode_step(dtype, q, k, v, log_a, beta, lambda, fenwick_states, t, out, B, H, dk, dv,
                                         Lmax, err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
}

int lla_debug_set_waits(int64_t limit_cycles, int hold) {
    if (current_device() < 0) return LLA_ERR_CUDA;
    return lla::tc_set_debug_waits(static_cast<long long>(limit_cycles), hold) == cudaSuccess ? LLA_OK : LLA_ERR_CUDA;
}

int lla_device_error(void* stream) {
    const int dev = current_device();
    if (dev < 0) return LLA_ERR_CUDA;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return LLA_ERR_CUDA;
    int word = 0;
    if (cudaMemcpyFromSymbol(&word, lla_device_error_word, sizeof(int)) != cudaSuccess) return LLA_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(lla_device_error_word, &zero, sizeof(int)) != cudaSuccess) return LLA_ERR_CUDA;
    if (word == lla::kDevBadInput) return LLA_ERR_DEVICE;
    if (word == lla::kDevTimeout) return LLA_ERR_TIMEOUT;
    return word == 0 ? LLA_OK : LLA_ERR_DEVICE;
}

}  // extern "C"
