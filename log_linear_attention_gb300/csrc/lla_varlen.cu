// Packed variable-length sequences: copies between the packed layout and the
// padded dense layout the prefill kernels take.
//
// Packed: every tensor is [H, total, W] row-major; sequence b owns the rows
// cu[b] .. cu[b+1]-1 of each head (cu = cu_seqlens, device int32 [n+1]), and
// each sequence's positions start at 0. Padded: [n, H, Tpad, Wp], sequence b of
// head h at (b * H + h), its first len_b rows copied, the rest zero; columns
// W..Wp-1 zero. Rows after a sequence's end are never reached by its causal
// outputs, so the dense prefill of the padded tensors gives every packed row
// exactly (up to rounding order) the output of its own sequence.
// A length outside [0, max_len] or a row range past `total` is recorded as bad
// input in the device error word and copies nothing.
#include "lla_internal.cuh"

namespace lla {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ bool seq_range(const int32_t* cu, int b, int total, int max_len, int& c0, int& len,
                                          int* err) {
    c0 = cu[b];
    const int c1 = cu[b + 1];
    if (c0 < 0 || c1 < c0 || c1 > total || c1 - c0 > max_len) {
        if (threadIdx.x == 0 && blockIdx.x == 0) record_error(err, kDevBadInput);
        len = 0;
        return false;
    }
    len = c1 - c0;
    return true;
}

// One warp per padded row: grid (ceil(Tpad / 8), n * H), 256 threads. Rows whose width
// is a multiple of 16 bytes (and no column padding) move as 16-byte vectors; others
// element by element.
template <typename E>
__global__ void __launch_bounds__(kThreads) pack_rows_kernel(const E* __restrict__ src, E* __restrict__ dst,
                                                             const int32_t* __restrict__ cu, int H, int total,
                                                             int Tpad, int W, int Wp, int max_len, int* err) {
    const int bh = blockIdx.y, b = bh / H, h = bh - b * H;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    int c0, len;
    seq_range(cu, b, total, max_len, c0, len, err);
    if (t >= Tpad) return;
    E* d = dst + (static_cast<size_t>(bh) * Tpad + t) * Wp;
    const E* s = src + (static_cast<size_t>(h) * total + c0 + t) * W;
    const bool live = t < len;
    if (W == Wp && (W * sizeof(E)) % 16 == 0) {
        const int nv = W * static_cast<int>(sizeof(E)) / 16;
        uint4* d4 = reinterpret_cast<uint4*>(d);
        const uint4* s4 = reinterpret_cast<const uint4*>(s);
        for (int c = lane; c < nv; c += 32) d4[c] = live ? s4[c] : make_uint4(0u, 0u, 0u, 0u);
    } else {
        for (int w = lane; w < Wp; w += 32) d[w] = (live && w < W) ? s[w] : E(0.f);
    }
}

// The inverse for the outputs: packed row cu[b] + t of head h <- padded row t of (b, h),
// t < len_b; same grid and vector rule.
template <typename E>
__global__ void __launch_bounds__(kThreads) unpack_rows_kernel(const E* __restrict__ src, E* __restrict__ dst,
                                                               const int32_t* __restrict__ cu, int H, int total,
                                                               int Tpad, int W, int max_len, int* err) {
    const int bh = blockIdx.y, b = bh / H, h = bh - b * H;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    int c0, len;
    seq_range(cu, b, total, max_len, c0, len, err);
    if (t >= len) return;
    const E* s = src + (static_cast<size_t>(bh) * Tpad + t) * W;
    E* d = dst + (static_cast<size_t>(h) * total + c0 + t) * W;
    if ((W * sizeof(E)) % 16 == 0) {
        const int nv = W * static_cast<int>(sizeof(E)) / 16;
        for (int c = lane; c < nv; c += 32) reinterpret_cast<uint4*>(d)[c] = reinterpret_cast<const uint4*>(s)[c];
    } else {
        for (int w = lane; w < W; w += 32) d[w] = s[w];
    }
}

template <typename E>
cudaError_t pack_t(const void* src, void* dst, const int32_t* cu, int n_seq, int H, int total, int Tpad, int W,
                   int Wp, int max_len, int* err, cudaStream_t stream) {
    if (n_seq * H > 65535) return cudaErrorInvalidValue;
    pack_rows_kernel<E><<<dim3((Tpad + 7) / 8, n_seq * H), kThreads, 0, stream>>>(
        static_cast<const E*>(src), static_cast<E*>(dst), cu, H, total, Tpad, W, Wp, max_len, err);
    return cudaGetLastError();
}

template <typename E>
cudaError_t unpack_t(const void* src, void* dst, const int32_t* cu, int n_seq, int H, int total, int Tpad, int W,
                     int max_len, int* err, cudaStream_t stream) {
    if (n_seq * H > 65535) return cudaErrorInvalidValue;
    unpack_rows_kernel<E><<<dim3((max_len + 7) / 8, n_seq * H), kThreads, 0, stream>>>(
        static_cast<const E*>(src), static_cast<E*>(dst), cu, H, total, Tpad, W, max_len, err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t varlen_pack(int elem_bytes, const void* src, void* dst, const int32_t* cu, int n_seq, int H, int total,
                        int Tpad, int W, int Wp, int max_len, int* err, cudaStream_t stream) {
    if (elem_bytes == 4)
        return pack_t<float>(src, dst, cu, n_seq, H, total, Tpad, W, Wp, max_len, err, stream);
    return pack_t<__nv_bfloat16>(src, dst, cu, n_seq, H, total, Tpad, W, Wp, max_len, err, stream);
}

cudaError_t varlen_unpack(int elem_bytes, const void* src, void* dst, const int32_t* cu, int n_seq, int H, int total,
                          int Tpad, int W, int max_len, int* err, cudaStream_t stream) {
    if (elem_bytes == 4) return unpack_t<float>(src, dst, cu, n_seq, H, total, Tpad, W, max_len, err, stream);
    return unpack_t<__nv_bfloat16>(src, dst, cu, n_seq, H, total, Tpad, W, max_len, err, stream);
}

}  // namespace lla
