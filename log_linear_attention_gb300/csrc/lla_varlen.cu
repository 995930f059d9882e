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
// input in the device error word; that sequence's padded rows are zero-filled and its
// packed output rows are not written.
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

// Each (sequence, head) is one contiguous block on both sides: the packed rows
// cu[b] .. cu[b+1]-1 of head h and the padded rows of (b, h). grid (x, n * H), 256 threads,
// grid-stride over the block. Where a row is a multiple of 16 bytes and is not widened, the
// copy moves 16-byte vectors; otherwise it walks the padded (row, column) elements.
constexpr int kUnitsPerThread = 4;

template <typename E>
__global__ void __launch_bounds__(kThreads) pack_rows_kernel(const E* __restrict__ src, E* __restrict__ dst,
                                                             const int32_t* __restrict__ cu, int H, int total,
                                                             int Tpad, int W, int Wp, int max_len, int* err) {
    const int bh = blockIdx.y, b = bh / H, h = bh - b * H;
    int c0, len;
    if (!seq_range(cu, b, total, max_len, c0, len, err)) c0 = 0;  // bad input: the block is zero-filled
    const size_t stride = static_cast<size_t>(gridDim.x) * kThreads;
    if (W == Wp && (W * sizeof(E)) % 16 == 0) {
        const size_t per_row = W * sizeof(E) / 16;
        const size_t n = static_cast<size_t>(Tpad) * per_row, live = static_cast<size_t>(len) * per_row;
        uint4* d = reinterpret_cast<uint4*>(dst) + static_cast<size_t>(bh) * n;
        const uint4* s = reinterpret_cast<const uint4*>(src) + (static_cast<size_t>(h) * total + c0) * per_row;
        for (size_t i = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x; i < n; i += stride)
            d[i] = i < live ? s[i] : make_uint4(0u, 0u, 0u, 0u);
    } else {
        const size_t n = static_cast<size_t>(Tpad) * Wp;
        E* d = dst + static_cast<size_t>(bh) * n;
        const E* s = src + (static_cast<size_t>(h) * total + c0) * W;
        for (size_t i = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x; i < n; i += stride) {
            const int t = static_cast<int>(i / Wp), w = static_cast<int>(i - static_cast<size_t>(t) * Wp);
            d[i] = (t < len && w < W) ? s[static_cast<size_t>(t) * W + w] : E(0.f);
        }
    }
}

// The inverse for the outputs: packed row cu[b] + t of head h <- padded row t of (b, h), t < len_b.
template <typename E>
__global__ void __launch_bounds__(kThreads) unpack_rows_kernel(const E* __restrict__ src, E* __restrict__ dst,
                                                               const int32_t* __restrict__ cu, int H, int total,
                                                               int Tpad, int W, int max_len, int* err) {
    const int bh = blockIdx.y, b = bh / H, h = bh - b * H;
    int c0, len;
    if (!seq_range(cu, b, total, max_len, c0, len, err)) return;
    const size_t stride = static_cast<size_t>(gridDim.x) * kThreads;
    if ((W * sizeof(E)) % 16 == 0) {
        const size_t per_row = W * sizeof(E) / 16, n = static_cast<size_t>(len) * per_row;
        const uint4* s = reinterpret_cast<const uint4*>(src) + static_cast<size_t>(bh) * Tpad * per_row;
        uint4* d = reinterpret_cast<uint4*>(dst) + (static_cast<size_t>(h) * total + c0) * per_row;
        for (size_t i = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x; i < n; i += stride) d[i] = s[i];
    } else {
        const size_t n = static_cast<size_t>(len) * W;
        const E* s = src + static_cast<size_t>(bh) * Tpad * W;
        E* d = dst + (static_cast<size_t>(h) * total + c0) * W;
        for (size_t i = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x; i < n; i += stride) d[i] = s[i];
    }
}

// CTAs per (sequence, head): enough for kUnitsPerThread units per thread over the padded block.
int blocks_per_seq(int Tpad, int W, int esz) {
    const size_t units = (W * esz) % 16 == 0 ? static_cast<size_t>(Tpad) * W * esz / 16 : static_cast<size_t>(Tpad) * W;
    const size_t per_block = static_cast<size_t>(kThreads) * kUnitsPerThread;
    const size_t nb = (units + per_block - 1) / per_block;
    return nb < 1 ? 1 : (nb > 1024 ? 1024 : static_cast<int>(nb));
}

template <typename E>
cudaError_t pack_t(const void* src, void* dst, const int32_t* cu, int n_seq, int H, int total, int Tpad, int W,
                   int Wp, int max_len, int* err, cudaStream_t stream) {
    if (n_seq * H > 65535) return cudaErrorInvalidValue;
    pack_rows_kernel<E><<<dim3(blocks_per_seq(Tpad, Wp, sizeof(E)), n_seq * H), kThreads, 0, stream>>>(
        static_cast<const E*>(src), static_cast<E*>(dst), cu, H, total, Tpad, W, Wp, max_len, err);
    return cudaGetLastError();
}

template <typename E>
cudaError_t unpack_t(const void* src, void* dst, const int32_t* cu, int n_seq, int H, int total, int Tpad, int W,
                     int max_len, int* err, cudaStream_t stream) {
    if (n_seq * H > 65535) return cudaErrorInvalidValue;
    unpack_rows_kernel<E><<<dim3(blocks_per_seq(max_len, W, sizeof(E)), n_seq * H), kThreads, 0, stream>>>(
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
