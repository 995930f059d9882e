// SIMT (CUDA-core, fp32 arithmetic) kernels of log-linear Mamba-2 attention.
//
// These run every shape the API accepts: the fp32 path (whose 1e-4 parity bar
// rules out TF32 tensor cores) and the bf16 shapes the tensor-core path does
// not cover. Chunkwise algorithm ("Log-Linear Attention", pt §2 "Forma
// Recorrente e Paralela" / fr §2 "Algorithmes Efficaces"): dense masked
// attention inside a chunk, plus, for every set bit p of the chunk index j, a
// read of the Fenwick node that sums the 2^p chunks before j's block boundary.
//
// Notation: C = chunk = 2^c, N = T / C chunks, g_i = sum of log_a over chunk i,
// cl_t = inclusive sum of log_a from the chunk start to t. Node (p, m) is
//   B_p[m] = sum_{s in chunks [m 2^p, (m+1) 2^p)} exp(decay from s to block end) k_s v_s^T
// and query t in chunk j reads, for each set bit p of j, node (p, (j >> p) - 1)
// weighted by lambda_t^(c+1+p) * exp(cl_t + sum_{i=(j>>p)<<p}^{j-1} g_i).
// Keys in that node are exactly those with 1 + floor(log2(t xor s)) = c+1+p.
#include "lla_internal.cuh"

namespace lla {
namespace {

constexpr int kThreads = 256;

// Inclusive prefix sum of n <= 128 values, by one warp (lane l owns 4 values).
__device__ void warp_scan128(const float* src, float* dst, int n) {
    const int lane = threadIdx.x & 31;
    float x[4];
    float run = 0.f;
#pragma unroll
    for (int e = 0; e < 4; e++) {
        int idx = lane * 4 + e;
        run += (idx < n) ? src[idx] : 0.f;
        x[e] = run;
    }
    float incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    float excl = incl - run;
#pragma unroll
    for (int e = 0; e < 4; e++) {
        int idx = lane * 4 + e;
        if (idx < n) dst[idx] = x[e] + excl;
    }
}

// g[bh][i] = sum of log_a over chunk i. One warp per chunk.
__global__ void __launch_bounds__(kThreads) chunk_totals_kernel(const float* __restrict__ log_a, float* __restrict__ g,
                                                                int T, int chunk, int N) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x * (kThreads / 32) + warp;
    const int bh = blockIdx.y;
    if (i >= N) return;
    const float* a = log_a + (size_t)bh * T + (size_t)i * chunk;
    float s = 0.f;
    for (int u = lane; u < chunk; u += 32) s += a[u];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) g[(size_t)bh * N + i] = s;
}

// Level-0 nodes: S_i = sum_{s in chunk i} exp(cl_end - cl_s) k_s v_s^T (fp32, [dk][dv]).
// grid (N, BH, ceil(dk*dv / 2048)); each thread owns 8 outputs.
template <typename T>
__global__ void __launch_bounds__(kThreads) chunk_state_kernel(const T* __restrict__ k, const T* __restrict__ v,
                                                               const float* __restrict__ log_a, float* __restrict__ nodes,
                                                               int Tlen, int dk, int dv, int chunk, int node_count) {
    __shared__ float araw[128], cl[128];
    __shared__ float ks[32][129];
    __shared__ float vs[32][128];
    const int tid = threadIdx.x;
    const int i = blockIdx.x, bh = blockIdx.y;
    const size_t s0 = (size_t)bh * Tlen + (size_t)i * chunk;
    for (int u = tid; u < chunk; u += kThreads) araw[u] = log_a[s0 + u];
    __syncthreads();
    if (tid < 32) warp_scan128(araw, cl, chunk);
    __syncthreads();
    const float cl_end = cl[chunk - 1];
    const int msz = dk * dv;
    float acc[8];
    int ei[8], en[8];
#pragma unroll
    for (int r = 0; r < 8; r++) {
        int e = blockIdx.z * 2048 + tid + r * kThreads;
        acc[r] = 0.f;
        ei[r] = (e < msz) ? e / dv : 0;
        en[r] = (e < msz) ? e % dv : 0;
    }
    for (int st = 0; st < chunk; st += 32) {
        const int ns = min(32, chunk - st);
        for (int x = tid; x < ns * dk; x += kThreads) {
            int sl = x / dk, d = x % dk;
            float w = expf(cl_end - cl[st + sl]);
            ks[sl][d] = w * load_f(k + (s0 + st + sl) * dk + d);
        }
        for (int x = tid; x < ns * dv; x += kThreads) {
            int sl = x / dv, n = x % dv;
            vs[sl][n] = load_f(v + (s0 + st + sl) * dv + n);
        }
        __syncthreads();
        for (int sl = 0; sl < ns; sl++) {
#pragma unroll
            for (int r = 0; r < 8; r++) acc[r] += ks[sl][ei[r]] * vs[sl][en[r]];
        }
        __syncthreads();
    }
    float* dst = nodes + ((size_t)bh * node_count + i) * msz;
#pragma unroll
    for (int r = 0; r < 8; r++) {
        int e = blockIdx.z * 2048 + tid + r * kThreads;
        if (e < msz) dst[e] = acc[r];
    }
}

struct LevelOffsets { int off[32]; };

// Pyramid levels 1..P-1: B_p[m] = exp(G_{p-1}[2m+1]) B_{p-1}[2m] + B_{p-1}[2m+1],
// G_p[m] = total log-decay of block (p, m). grid (ceil(dk*dv/256), BH); each thread
// owns one matrix element across all nodes of its head.
__global__ void __launch_bounds__(kThreads) pyramid_kernel(float* __restrict__ nodes, const float* __restrict__ g,
                                                           int N, int P, int node_count, int msz, LevelOffsets lo) {
    extern __shared__ float G[];  // node_count floats, same indexing as the nodes
    const int bh = blockIdx.y;
    for (int m = threadIdx.x; m < N; m += kThreads) G[m] = g[(size_t)bh * N + m];
    __syncthreads();
    for (int p = 1; p < P; p++) {
        for (int m = threadIdx.x; m < (N >> p); m += kThreads)
            G[lo.off[p] + m] = G[lo.off[p - 1] + 2 * m] + G[lo.off[p - 1] + 2 * m + 1];
        __syncthreads();
    }
    const int e = blockIdx.x * kThreads + threadIdx.x;
    if (e >= msz) return;
    float* base = nodes + (size_t)bh * node_count * msz + e;
    for (int p = 1; p < P; p++) {
        for (int m = 0; m < (N >> p); m++) {
            float lo_node = base[(size_t)(lo.off[p - 1] + 2 * m) * msz];
            float hi_node = base[(size_t)(lo.off[p - 1] + 2 * m + 1) * msz];
            base[(size_t)(lo.off[p] + m) * msz] = expf(G[lo.off[p - 1] + 2 * m + 1]) * lo_node + hi_node;
        }
    }
}

// Output for 16 queries per block: intra-chunk masked attention plus the
// lambda-weighted Fenwick node reads. grid (T/16, BH).
template <typename T>
__global__ void __launch_bounds__(kThreads) output_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                          const T* __restrict__ v, const float* __restrict__ log_a,
                                                          const float* __restrict__ lambda, const float* __restrict__ g,
                                                          const float* __restrict__ nodes, T* __restrict__ out,
                                                          int Tlen, int dk, int dv, int chunk, int c, int N, int L,
                                                          int P, int node_count, LevelOffsets lo) {
    __shared__ float qs[16][129];
    __shared__ float araw[128], cl[128];
    __shared__ float lam[16][33];
    __shared__ float ks[32][129];
    __shared__ float vs[32][128];
    __shared__ float ps[16][33];
    __shared__ float rp[16];
    __shared__ float dsum;
    const int tid = threadIdx.x;
    const int bh = blockIdx.y;
    const int t0 = blockIdx.x * 16;
    const int j = t0 >> c;
    const int c0 = j << c;
    const size_t row0 = (size_t)bh * Tlen;

    for (int x = tid; x < 16 * dk; x += kThreads) qs[x / dk][x % dk] = load_f(q + (row0 + t0 + x / dk) * dk + x % dk);
    for (int x = tid; x < 16 * L; x += kThreads) lam[x / L][x % L] = lambda[(row0 + t0 + x / L) * L + x % L];
    for (int u = tid; u < chunk; u += kThreads) araw[u] = log_a[row0 + c0 + u];
    __syncthreads();
    if (tid < 32) warp_scan128(araw, cl, chunk);
    __syncthreads();

    float acc[8];
    int oq[8], on[8];
    const int nout = 16 * dv;
#pragma unroll
    for (int r = 0; r < 8; r++) {
        int o = tid + r * kThreads;
        acc[r] = 0.f;
        oq[r] = (o < nout) ? o / dv : 0;
        on[r] = (o < nout) ? o % dv : 0;
    }

    // Intra-chunk: keys from the chunk start up to the last query of this block.
    for (int st = c0; st < t0 + 16; st += 32) {
        const int nk = min(32, t0 + 16 - st);
        for (int x = tid; x < nk * dk; x += kThreads) ks[x / dk][x % dk] = load_f(k + (row0 + st + x / dk) * dk + x % dk);
        for (int x = tid; x < nk * dv; x += kThreads) vs[x / dv][x % dv] = load_f(v + (row0 + st + x / dv) * dv + x % dv);
        __syncthreads();
        for (int pr = tid; pr < 16 * 32; pr += kThreads) {
            const int tq = pr >> 5, sl = pr & 31;
            const int t = t0 + tq, s = st + sl;
            float val = 0.f;
            if (sl < nk && s <= t) {
                float dot = 0.f;
                for (int d = 0; d < dk; d++) dot += qs[tq][d] * ks[sl][d];
                val = dot * expf(cl[t - c0] - cl[s - c0]) * lam[tq][fenwick_level(t, s)];
            }
            ps[tq][sl] = val;
        }
        __syncthreads();
        for (int sl = 0; sl < nk; sl++) {
#pragma unroll
            for (int r = 0; r < 8; r++) acc[r] += ps[oq[r]][sl] * vs[sl][on[r]];
        }
        __syncthreads();
    }

    // Inter-chunk: one Fenwick node per set bit p of the chunk index.
    for (int p = 0; p < P; p++) {
        if (((j >> p) & 1) == 0) continue;
        const int m = (j >> p) - 1;
        if (tid < 32) {
            float d = 0.f;
            for (int i = ((j >> p) << p) + tid; i < j; i += 32) d += g[(size_t)bh * N + i];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
            if (tid == 0) dsum = d;
        }
        __syncthreads();
        if (tid < 16) rp[tid] = lam[tid][c + 1 + p] * expf(cl[t0 + tid - c0] + dsum);
        const float* node = nodes + ((size_t)bh * node_count + lo.off[p] + m) * (size_t)(dk * dv);
        float tmp[8];
#pragma unroll
        for (int r = 0; r < 8; r++) tmp[r] = 0.f;
        for (int it = 0; it < dk; it += 32) {
            const int ni = min(32, dk - it);
            __syncthreads();
            for (int x = tid; x < ni * dv; x += kThreads) vs[x / dv][x % dv] = node[(size_t)(it + x / dv) * dv + x % dv];
            __syncthreads();
            for (int il = 0; il < ni; il++) {
#pragma unroll
                for (int r = 0; r < 8; r++) tmp[r] += qs[oq[r]][it + il] * vs[il][on[r]];
            }
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < 8; r++) acc[r] += rp[oq[r]] * tmp[r];
        __syncthreads();
    }

#pragma unroll
    for (int r = 0; r < 8; r++) {
        int o = tid + r * kThreads;
        if (o < nout) store_f(out + (row0 + t0 + oq[r]) * dv + on[r], acc[r]);
    }
}

// One decode step per (b, h); see lla_decode_step in include/lla.h.
// Thread layout: float4 column group col4 = tid % DV4 (fixed per thread), rows
// i = tid / DV4 + r * (256 / DV4). Each state element is read once and written once.
template <typename T, int DV4>
__global__ void __launch_bounds__(kThreads) decode_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                          const T* __restrict__ v, const float* __restrict__ log_a,
                                                          const float* __restrict__ lambda, float* __restrict__ states,
                                                          const int64_t* __restrict__ tpos, T* __restrict__ out,
                                                          int H, int dk, int Lmax, int* err) {
    constexpr int DV = DV4 * 4;
    constexpr int ROWS_PER_PASS = kThreads / DV4;
    __shared__ float qsh[256], ksh[256];
    __shared__ float vsh[DV];
    __shared__ float lam[40];
    __shared__ float red[kThreads / 32][DV];
    const int tid = threadIdx.x;
    const int bh = blockIdx.x;
    const int b = bh / H;
    const int64_t tb = tpos[b];
    if (tb < 0 || tb >= ((int64_t)1 << (Lmax - 1))) {
        if (tid == 0) record_error(err, kDevBadInput);
        return;
    }
    for (int x = tid; x < dk; x += kThreads) {
        qsh[x] = load_f(q + (size_t)bh * dk + x);
        ksh[x] = load_f(k + (size_t)bh * dk + x);
    }
    for (int x = tid; x < DV; x += kThreads) vsh[x] = load_f(v + (size_t)bh * DV + x);
    for (int x = tid; x < Lmax; x += kThreads) lam[x] = lambda[(size_t)bh * Lmax + x];
    __syncthreads();

    const float a = expf(log_a[bh]);
    const int c = tb > 0 ? __ffsll((long long)tb) - 1 : -1;  // trailing zeros of t
    const int top = tb > 0 ? 64 - __clzll((long long)tb) : 0;  // bitlength(t): highest nonempty level
    const int col4 = tid % DV4;
    const size_t msz4 = (size_t)dk * DV4;
    float4* S = reinterpret_cast<float4*>(states) + (size_t)bh * Lmax * msz4;
    const float4 v4 = make_float4(vsh[col4 * 4], vsh[col4 * 4 + 1], vsh[col4 * 4 + 2], vsh[col4 * 4 + 3]);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);

    for (int i = tid / DV4; i < dk; i += ROWS_PER_PASS) {
        const size_t e = (size_t)i * DV4 + col4;
        const float qi = qsh[i];
        if (tb > 0) {
            // levels 0..c (all held for t-1) merge into level c+1, decayed by a_t
            float4 mrg = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int l = 0; l <= c; l++) {
                float4 x = S[l * msz4 + e];
                mrg.x += x.x; mrg.y += x.y; mrg.z += x.z; mrg.w += x.w;
            }
            mrg.x *= a; mrg.y *= a; mrg.z *= a; mrg.w *= a;
            S[(c + 1) * msz4 + e] = mrg;
            const float wq = lam[c + 1] * qi;
            o.x += wq * mrg.x; o.y += wq * mrg.y; o.z += wq * mrg.z; o.w += wq * mrg.w;
            // coarser levels held for both t-1 and t: decay in place
            for (int l = c + 2; l <= top; l++) {
                if (((tb >> (l - 1)) & 1) == 0) continue;
                float4 x = S[l * msz4 + e];
                x.x *= a; x.y *= a; x.z *= a; x.w *= a;
                S[l * msz4 + e] = x;
                const float w = lam[l] * qi;
                o.x += w * x.x; o.y += w * x.y; o.z += w * x.z; o.w += w * x.w;
            }
        }
        // level 0: the new token
        const float ki = ksh[i];
        const float4 x0 = make_float4(ki * v4.x, ki * v4.y, ki * v4.z, ki * v4.w);
        S[e] = x0;
        const float w0 = lam[0] * qi;
        o.x += w0 * x0.x; o.y += w0 * x0.y; o.z += w0 * x0.z; o.w += w0 * x0.w;
    }

    // reduce over rows: lanes with equal col4 inside a warp, then across warps
#pragma unroll
    for (int off = DV4; off < 32; off <<= 1) {
        o.x += __shfl_xor_sync(0xffffffffu, o.x, off);
        o.y += __shfl_xor_sync(0xffffffffu, o.y, off);
        o.z += __shfl_xor_sync(0xffffffffu, o.z, off);
        o.w += __shfl_xor_sync(0xffffffffu, o.w, off);
    }
    const int warp = tid >> 5, lane = tid & 31;
    if (lane < DV4) {
        red[warp][lane * 4 + 0] = o.x;
        red[warp][lane * 4 + 1] = o.y;
        red[warp][lane * 4 + 2] = o.z;
        red[warp][lane * 4 + 3] = o.w;
    }
    __syncthreads();
    if (tid < DV) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; w++) s += red[w][tid];
        store_f(out + (size_t)bh * DV + tid, s);
    }
}

// The decode step for dk = DK known at compile time: each thread owns column group
// col4 and rows i = tid / DV4 + r * (256 / DV4), r < RPT. Levels are the outer loop
// and a thread's RPT rows are unrolled inside it, so every level issues RPT
// independent 128-bit loads per thread. The state stream bypasses L2 retention
// (evict-first loads and stores): it is read once and written once per step.
template <typename T, int DV4, int DK>
__global__ void __launch_bounds__(kThreads) decode_kernel_fixed(const T* __restrict__ q, const T* __restrict__ k,
                                                                const T* __restrict__ v, const float* __restrict__ log_a,
                                                                const float* __restrict__ lambda,
                                                                float* __restrict__ states,
                                                                const int64_t* __restrict__ tpos, T* __restrict__ out,
                                                                int H, int Lmax, int* err) {
    constexpr int DV = DV4 * 4;
    constexpr int ROWS_PER_PASS = kThreads / DV4;
    constexpr int RPT = DK / ROWS_PER_PASS;
    static_assert(DK % ROWS_PER_PASS == 0, "rows must divide evenly");
    __shared__ float qsh[DK], ksh[DK];
    __shared__ float vsh[DV];
    __shared__ float lam[40];
    __shared__ float red[kThreads / 32][DV];
    const int tid = threadIdx.x;
    const int bh = blockIdx.x;
    const int b = bh / H;
    const int64_t tb = tpos[b];
    if (tb < 0 || tb >= ((int64_t)1 << (Lmax - 1))) {
        if (tid == 0) record_error(err, kDevBadInput);
        return;
    }
    for (int x = tid; x < DK; x += kThreads) {
        qsh[x] = load_f(q + (size_t)bh * DK + x);
        ksh[x] = load_f(k + (size_t)bh * DK + x);
    }
    for (int x = tid; x < DV; x += kThreads) vsh[x] = load_f(v + (size_t)bh * DV + x);
    for (int x = tid; x < Lmax; x += kThreads) lam[x] = lambda[(size_t)bh * Lmax + x];
    __syncthreads();

    const float a = expf(log_a[bh]);
    const int c = tb > 0 ? __ffsll((long long)tb) - 1 : -1;  // trailing zeros of t
    const int top = tb > 0 ? 64 - __clzll((long long)tb) : 0;  // bitlength(t): highest nonempty level
    const int col4 = tid % DV4;
    const int row0 = tid / DV4;
    constexpr size_t msz4 = (size_t)DK * DV4;
    float4* S = reinterpret_cast<float4*>(states) + (size_t)bh * Lmax * msz4 + (size_t)row0 * DV4 + col4;
    constexpr size_t rstep = (size_t)ROWS_PER_PASS * DV4;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);

    if (tb > 0) {
        // levels 0..c (all held for t-1) merge into level c+1, decayed by a_t
        float4 mrg[RPT];
#pragma unroll
        for (int r = 0; r < RPT; r++) mrg[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int l = 0; l <= c; l++) {
            float4 x[RPT];
#pragma unroll
            for (int r = 0; r < RPT; r++) x[r] = __ldcs(S + l * msz4 + r * rstep);
#pragma unroll
            for (int r = 0; r < RPT; r++) {
                mrg[r].x += x[r].x; mrg[r].y += x[r].y; mrg[r].z += x[r].z; mrg[r].w += x[r].w;
            }
        }
        const float lc = lam[c + 1];
#pragma unroll
        for (int r = 0; r < RPT; r++) {
            float4 m = mrg[r];
            m.x *= a; m.y *= a; m.z *= a; m.w *= a;
            __stcs(S + (c + 1) * msz4 + r * rstep, m);
            const float wq = lc * qsh[row0 + r * ROWS_PER_PASS];
            o.x += wq * m.x; o.y += wq * m.y; o.z += wq * m.z; o.w += wq * m.w;
        }
        // coarser levels held for both t-1 and t: decay in place
        for (int l = c + 2; l <= top; l++) {
            if (((tb >> (l - 1)) & 1) == 0) continue;
            float4 x[RPT];
#pragma unroll
            for (int r = 0; r < RPT; r++) x[r] = __ldcs(S + l * msz4 + r * rstep);
            const float ll = lam[l];
#pragma unroll
            for (int r = 0; r < RPT; r++) {
                x[r].x *= a; x[r].y *= a; x[r].z *= a; x[r].w *= a;
                __stcs(S + l * msz4 + r * rstep, x[r]);
                const float w = ll * qsh[row0 + r * ROWS_PER_PASS];
                o.x += w * x[r].x; o.y += w * x[r].y; o.z += w * x[r].z; o.w += w * x[r].w;
            }
        }
    }
    // level 0: the new token
    {
        const float4 v4 = make_float4(vsh[col4 * 4], vsh[col4 * 4 + 1], vsh[col4 * 4 + 2], vsh[col4 * 4 + 3]);
        const float l0 = lam[0];
#pragma unroll
        for (int r = 0; r < RPT; r++) {
            const int i = row0 + r * ROWS_PER_PASS;
            const float ki = ksh[i];
            const float4 x0 = make_float4(ki * v4.x, ki * v4.y, ki * v4.z, ki * v4.w);
            __stcs(S + r * rstep, x0);
            const float w0 = l0 * qsh[i];
            o.x += w0 * x0.x; o.y += w0 * x0.y; o.z += w0 * x0.z; o.w += w0 * x0.w;
        }
    }

#pragma unroll
    for (int off = DV4; off < 32; off <<= 1) {
        o.x += __shfl_xor_sync(0xffffffffu, o.x, off);
        o.y += __shfl_xor_sync(0xffffffffu, o.y, off);
        o.z += __shfl_xor_sync(0xffffffffu, o.z, off);
        o.w += __shfl_xor_sync(0xffffffffu, o.w, off);
    }
    const int warp = tid >> 5, lane = tid & 31;
    if (lane < DV4) {
        red[warp][lane * 4 + 0] = o.x;
        red[warp][lane * 4 + 1] = o.y;
        red[warp][lane * 4 + 2] = o.z;
        red[warp][lane * 4 + 3] = o.w;
    }
    __syncthreads();
    if (tid < DV) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; w++) sum += red[w][tid];
        store_f(out + (size_t)bh * DV + tid, sum);
    }
}

// ---- state set after a prefill (hand-off to the decode step)

// Where the rows of sequence bh start and how many there are: every sequence has T rows
// at bh * T (dense), or, with cu_seqlens, sequence b of head h has cu[b+1] - cu[b] rows
// starting at h * total + cu[b] (packed). A packed length outside [0, T] or past
// `total` is reported as bad input and treated as empty.
struct SeqRows {
    const int32_t* cu;
    int T, H, total;
    __device__ bool get(int bh, size_t& base, int& len, int* err) const {
        if (!cu) {
            base = static_cast<size_t>(bh) * T;
            len = T;
            return true;
        }
        const int b = bh / H, h = bh - b * H;
        const int c0 = cu[b], c1 = cu[b + 1];
        if (c0 < 0 || c1 < c0 || c1 > total || c1 - c0 > T) {
            if (threadIdx.x == 0) record_error(err, kDevBadInput);
            base = 0;
            len = 0;
            return false;
        }
        base = static_cast<size_t>(h) * total + c0;
        len = c1 - c0;
        return true;
    }
};

// Per sequence: the decay exponent from each token s to the last token pos = len-1,
// suf[base + s] = sum_{r=s+1..pos} log_a_r, accumulated from pos downwards (so the
// values near pos, the ones that matter, carry the least rounding); also writes
// slot 0 (k_pos v_pos^T) and zeroes the other slots the pieces add into.
// grid (sequences x heads), 256 threads.
template <typename T>
__global__ void __launch_bounds__(kThreads) state_scan_kernel(const T* __restrict__ k, const T* __restrict__ v,
                                                              const float* __restrict__ log_a, float* __restrict__ suf,
                                                              float* __restrict__ states, SeqRows rows, int dk, int dv,
                                                              int Lmax, int* err) {
    __shared__ float carry_sh;
    __shared__ float tile[kThreads];
    const int bh = blockIdx.x, tid = threadIdx.x;
    size_t base;
    int len;
    rows.get(bh, base, len, err);
    if (len == 0) return;  // an empty sequence holds no slot
    const float* a = log_a + base;
    float* sf = suf + base;
    const int pos = len - 1;
    if (tid == 0) carry_sh = 0.f;
    __syncthreads();
    // blocks of 256 tokens from the end: suf[s] = carry + sum_{r in (s, block end]} log_a_r
    for (int end = pos; end >= 0; end -= kThreads) {
        const int s = end - tid;
        // inclusive suffix within the block of a[s+1 .. end]: x_s = a[s+1] (0 for s = pos)
        tile[tid] = (s >= 0 && s + 1 <= pos) ? a[s + 1] : 0.f;
        __syncthreads();
        // Hillis-Steele inclusive scan over tid (tid 0 = the block's last token)
        for (int off = 1; off < kThreads; off <<= 1) {
            const float y = tid >= off ? tile[tid - off] : 0.f;
            __syncthreads();
            tile[tid] += y;
            __syncthreads();
        }
        const float carry = carry_sh;
        if (s >= 0) sf[s] = carry + tile[tid];
        __syncthreads();
        if (tid == kThreads - 1) carry_sh = carry + tile[tid];
        __syncthreads();
    }
    const size_t msz = (size_t)dk * dv;
    float* st = states + (size_t)bh * Lmax * msz;
    for (int l = 1; l < Lmax; l++) {
        if (l - 1 >= 31 || ((pos >> (l - 1)) & 1) == 0) continue;
        for (size_t e = tid; e < msz; e += kThreads) st[l * msz + e] = 0.f;
    }
    const size_t r = base + pos;
    for (size_t e = tid; e < msz; e += kThreads)
        st[e] = load_f(k + r * dk + e / dv) * load_f(v + r * dv + e % dv);
}

constexpr int kPieceLen = 512;

// Piece idx of pos's Fenwick walk: buckets [b - lowbit(b), b) from b = pos down, each cut
// into pieces of at most kPieceLen keys. Returns false when idx is past the last piece.
__device__ bool fenwick_piece(int pos, int idx, int& level, int& s0, int& s1) {
    int n = 0;
    for (int b = pos; b > 0; b -= b & (-b)) {
        const int low = b & (-b);
        const int np = (low + kPieceLen - 1) / kPieceLen;
        if (idx < n + np) {
            level = 32 - __clz(low);  // log2(low) + 1
            s0 = b - low + (idx - n) * kPieceLen;
            s1 = min(s0 + kPieceLen, b);
            return true;
        }
        n += np;
    }
    return false;
}

// One piece [start, end) of a Fenwick bucket of pos = len-1: adds
// sum_s exp(suf[s]) k_s v_s^T into its slot. grid (pieces, sequences x heads, ceil(dk*dv / 2048)).
template <typename T>
__global__ void __launch_bounds__(kThreads) state_piece_kernel(const T* __restrict__ k, const T* __restrict__ v,
                                                               const float* __restrict__ suf, float* __restrict__ states,
                                                               SeqRows rows, int dk, int dv, int Lmax, int* err) {
    __shared__ float ks[32][129];
    __shared__ float vs[32][128];
    const int tid = threadIdx.x;
    const int bh = blockIdx.y;
    size_t row0;
    int len;
    rows.get(bh, row0, len, err);
    int l, s0, s1;
    if (len < 2 || !fenwick_piece(len - 1, blockIdx.x, l, s0, s1)) return;
    const int msz = dk * dv;
    float acc[8];
    int ei[8], en[8];
#pragma unroll
    for (int r = 0; r < 8; r++) {
        const int e = blockIdx.z * 2048 + tid + r * kThreads;
        acc[r] = 0.f;
        ei[r] = (e < msz) ? e / dv : 0;
        en[r] = (e < msz) ? e % dv : 0;
    }
    for (int st = s0; st < s1; st += 32) {
        const int ns = min(32, s1 - st);
        for (int x = tid; x < ns * dk; x += kThreads) {
            const int sl = x / dk, d = x % dk;
            ks[sl][d] = expf(suf[row0 + st + sl]) * load_f(k + (row0 + st + sl) * dk + d);
        }
        for (int x = tid; x < ns * dv; x += kThreads) vs[x / dv][x % dv] = load_f(v + (row0 + st + x / dv) * dv + x % dv);
        __syncthreads();
        for (int sl = 0; sl < ns; sl++) {
#pragma unroll
            for (int r = 0; r < 8; r++) acc[r] += ks[sl][ei[r]] * vs[sl][en[r]];
        }
        __syncthreads();
    }
    float* dst = states + ((size_t)bh * Lmax + l) * msz;
#pragma unroll
    for (int r = 0; r < 8; r++) {
        const int e = blockIdx.z * 2048 + tid + r * kThreads;
        if (e < msz) atomicAdd(dst + e, acc[r]);
    }
}

template <typename T>
cudaError_t prefill_state_t(const void* k, const void* v, const float* log_a, float* states, int n_seq, int H,
                            SeqRows rows, int dk, int dv, int Lmax, void* workspace, int* err, cudaStream_t stream) {
    const int BH = n_seq * H;
    float* suf = static_cast<float*>(workspace);
    // pieces of the longest walk: at most T / kPieceLen whole pieces plus one per bucket
    const int max_pieces = rows.T / kPieceLen + 32;
    state_scan_kernel<T><<<BH, kThreads, 0, stream>>>(static_cast<const T*>(k), static_cast<const T*>(v), log_a, suf,
                                                       states, rows, dk, dv, Lmax, err);
    note_launch(stream, "state_scan");
    state_piece_kernel<T><<<dim3(max_pieces, BH, (dk * dv + 2047) / 2048), kThreads, 0, stream>>>(
        static_cast<const T*>(k), static_cast<const T*>(v), suf, states, rows, dk, dv, Lmax, err);
    note_launch(stream, "state_pieces");
    return cudaGetLastError();
}

template <typename T>
cudaError_t simt_nodes_t(const SimtPlan& pl, const T* k, const T* v, const float* log_a, void* workspace,
                         cudaStream_t stream) {
    const int BH = pl.B * pl.H;
    float* g = reinterpret_cast<float*>(workspace);
    float* nodes = reinterpret_cast<float*>(reinterpret_cast<char*>(workspace) + pl.g_bytes);
    LevelOffsets lo;
    for (int p = 0; p < 32; p++) lo.off[p] = pl.level_off[p];
    chunk_totals_kernel<<<dim3((pl.N + 7) / 8, BH), kThreads, 0, stream>>>(log_a, g, pl.T, pl.chunk, pl.N);
    const int msz = pl.dk * pl.dv;
    if (pl.P > 0)
        chunk_state_kernel<T><<<dim3(pl.N, BH, (msz + 2047) / 2048), kThreads, 0, stream>>>(k, v, log_a, nodes, pl.T,
                                                                                           pl.dk, pl.dv, pl.chunk,
                                                                                           pl.node_count);
    if (pl.P > 1)
        pyramid_kernel<<<dim3((msz + kThreads - 1) / kThreads, BH), kThreads, pl.node_count * sizeof(float), stream>>>(
            nodes, g, pl.N, pl.P, pl.node_count, msz, lo);
    return cudaGetLastError();
}

template <typename T>
cudaError_t simt_forward_t(const SimtPlan& pl, const T* q, const T* k, const T* v, const float* log_a,
                           const float* lambda, T* out, void* workspace, cudaStream_t stream) {
    const int BH = pl.B * pl.H;
    float* g = reinterpret_cast<float*>(workspace);
    float* nodes = reinterpret_cast<float*>(reinterpret_cast<char*>(workspace) + pl.g_bytes);
    LevelOffsets lo;
    for (int p = 0; p < 32; p++) lo.off[p] = pl.level_off[p];
    const int L = bitlength((int64_t)pl.T - 1) + 1;
    chunk_totals_kernel<<<dim3((pl.N + 7) / 8, BH), kThreads, 0, stream>>>(log_a, g, pl.T, pl.chunk, pl.N);
    note_launch(stream, "simt_chunk_totals");
    if (pl.P > 0) {
        const int msz = pl.dk * pl.dv;
        chunk_state_kernel<T><<<dim3(pl.N, BH, (msz + 2047) / 2048), kThreads, 0, stream>>>(
            k, v, log_a, nodes, pl.T, pl.dk, pl.dv, pl.chunk, pl.node_count);
        note_launch(stream, "simt_chunk_state");
        if (pl.P > 1)
            pyramid_kernel<<<dim3((msz + kThreads - 1) / kThreads, BH), kThreads, pl.node_count * sizeof(float),
                             stream>>>(nodes, g, pl.N, pl.P, pl.node_count, msz, lo);
        if (pl.P > 1) note_launch(stream, "simt_pyramid");
    }
    output_kernel<T><<<dim3(pl.T / 16, BH), kThreads, 0, stream>>>(q, k, v, log_a, lambda, g, nodes, out, pl.T,
                                                                    pl.dk, pl.dv, pl.chunk, pl.c, pl.N, L, pl.P,
                                                                    pl.node_count, lo);
    note_launch(stream, "simt_output");
    return cudaGetLastError();
}

template <typename T, int DV4>
void launch_decode(const void* q, const void* k, const void* v, const float* log_a, const float* lambda,
                   float* states, const int64_t* t, void* out, int B, int H, int dk, int Lmax, int* err,
                   cudaStream_t stream) {
    if (dk == 128) {
        decode_kernel_fixed<T, DV4, 128><<<B * H, kThreads, 0, stream>>>(
            static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), log_a, lambda, states, t,
            static_cast<T*>(out), H, Lmax, err);
        note_launch(stream, "decode_step");
        return;
    }
    decode_kernel<T, DV4><<<B * H, kThreads, 0, stream>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), log_a, lambda, states, t,
        static_cast<T*>(out), H, dk, Lmax, err);
    note_launch(stream, "decode_step");
}

template <typename T>
cudaError_t decode_t(const void* q, const void* k, const void* v, const float* log_a, const float* lambda,
                     float* states, const int64_t* t, void* out, int B, int H, int dk, int dv, int Lmax, int* err,
                     cudaStream_t stream) {
    switch (dv) {
        case 16: launch_decode<T, 4>(q, k, v, log_a, lambda, states, t, out, B, H, dk, Lmax, err, stream); break;
        case 32: launch_decode<T, 8>(q, k, v, log_a, lambda, states, t, out, B, H, dk, Lmax, err, stream); break;
        case 64: launch_decode<T, 16>(q, k, v, log_a, lambda, states, t, out, B, H, dk, Lmax, err, stream); break;
        case 128: launch_decode<T, 32>(q, k, v, log_a, lambda, states, t, out, B, H, dk, Lmax, err, stream); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

bool make_simt_plan(int B, int H, int T, int dk, int dv, int chunk, SimtPlan* pl) {
    pl->B = B; pl->H = H; pl->T = T; pl->dk = dk; pl->dv = dv; pl->chunk = chunk;
    pl->c = bitlength(chunk) - 1;
    pl->N = T / chunk;
    pl->P = bitlength((int64_t)pl->N - 1);
    int off = 0;
    for (int p = 0; p < 32; p++) {
        pl->level_off[p] = off;
        if (p < pl->P) off += pl->N >> p;
    }
    pl->node_count = off;
    // the pyramid kernel keeps one fp32 block-decay total per node in shared memory
    if (pl->node_count > 12288) return false;
    const size_t BH = (size_t)B * H;
    pl->g_bytes = ((BH * pl->N * sizeof(float)) + 255) / 256 * 256;
    pl->nodes_bytes = BH * (size_t)pl->node_count * dk * dv * sizeof(float);
    pl->total_bytes = pl->g_bytes + pl->nodes_bytes;
    return true;
}

cudaError_t simt_forward(const SimtPlan& pl, int dtype, const void* q, const void* k, const void* v,
                         const float* log_a, const float* lambda, void* out, void* workspace, int* err,
                         cudaStream_t stream) {
    (void)err;
    if (dtype == 1)
        return simt_forward_t<float>(pl, static_cast<const float*>(q), static_cast<const float*>(k),
                                     static_cast<const float*>(v), log_a, lambda, static_cast<float*>(out),
                                     workspace, stream);
    return simt_forward_t<__nv_bfloat16>(pl, static_cast<const __nv_bfloat16*>(q),
                                         static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v),
                                         log_a, lambda, static_cast<__nv_bfloat16*>(out), workspace, stream);
}

cudaError_t simt_nodes(const SimtPlan& pl, int dtype, const void* k, const void* v, const float* log_a,
                       void* workspace, cudaStream_t stream) {
    if (dtype == 1)
        return simt_nodes_t<float>(pl, static_cast<const float*>(k), static_cast<const float*>(v), log_a, workspace,
                                   stream);
    return simt_nodes_t<__nv_bfloat16>(pl, static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v),
                                       log_a, workspace, stream);
}

cudaError_t prefill_state(int dtype, const void* k, const void* v, const float* log_a, float* states, int B, int H,
                          int T, int dk, int dv, int Lmax, void* workspace, int* err, cudaStream_t stream,
                          const int32_t* cu_seqlens, int total) {
    SeqRows rows{cu_seqlens, T, H, total};
    if (dtype == 1)
        return prefill_state_t<float>(k, v, log_a, states, B, H, rows, dk, dv, Lmax, workspace, err, stream);
    return prefill_state_t<__nv_bfloat16>(k, v, log_a, states, B, H, rows, dk, dv, Lmax, workspace, err, stream);
}

cudaError_t decode_step(int dtype, const void* q, const void* k, const void* v, const float* log_a,
                        const float* lambda, float* states, const int64_t* t, void* out, int B, int H, int dk,
                        int dv, int Lmax, int* err, cudaStream_t stream) {
    if (dtype == 1) return decode_t<float>(q, k, v, log_a, lambda, states, t, out, B, H, dk, dv, Lmax, err, stream);
    return decode_t<__nv_bfloat16>(q, k, v, log_a, lambda, states, t, out, B, H, dk, dv, Lmax, err, stream);
}

}  // namespace lla
