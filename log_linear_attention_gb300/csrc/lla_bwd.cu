// Backward pass of causal log-linear Mamba-2 attention (CUDA cores, fp32 arithmetic).
//
// For an upstream gradient dO and the loss L = sum_t dO_t . o_t, with
//   o_t = sum_{s<=t} lambda_t^(l(t,s)) exp(cum_t - cum_s) (q_t . k_s) v_s
// ("Log-Linear Attention", pt §2 "Mascara Hierarquica" / fr §2 "Matrice de
// Masque Hierarchique" for the operator, pt §2 "Forma Recorrente e Paralela" /
// fr §2 "Algorithmes Efficaces" for the chunkwise form whose backward this is),
// the gradients follow the forward's chunkwise structure. Notation: C = chunk,
// N = T / C chunks, node (p, m) = B_{p,m} = sum over the keys of chunks
// [m 2^p, (m+1) 2^p) of exp(decay to the block end e) k_s v_s^T; chunk j
// reads node (p, (j >> p) - 1) for each set bit p of j, weighted per query by
// r_{t,p} = lambda_t^(c+1+p) exp(cum_t - cum_e).
//
//   * Node gradients: dB_{p,m} = sum over the query block that reads it,
//     chunks [(m+1) 2^p, (m+2) 2^p), of r_{t,p} q_t dO_t^T   (bwd_dnode).
//   * Key side: a key chunk i sits in node (p, i >> p) at every level; the
//     read ones combine into C_i = sum_p exp(cum_{e_p} - cum_{end_i}) dB_{p,i>>p},
//     computed top-down like a transposed pyramid (bwd_topdown_level, in place
//     over the dB array, so level 0 ends holding C_i). Then for s in chunk i,
//     with w_s = exp(cum_{end_i} - cum_s): dk_s += w_s C_i v_s,
//     dv_s += w_s C_i^T k_s.
//   * Query side: dq_t += sum_p r_{t,p} B_{p,m} dO_t, and
//     dlambda_t^(c+1+p) = exp(cum_t - cum_e) q_t^T B_{p,m} dO_t.
//   * Inside a chunk every pair is dense: with A_ts = lambda D qk and
//     G_ts = lambda D (dO_t . v_s): dq = G K, dk = G^T Q, dv = A^T dO,
//     dlambda_t^(l) += D qk (dO_t . v_s) for the pair's level l <= c.
//   * Decay: each pair's term depends on cum_t - cum_s only; its derivative
//     E_ts = lambda D qk (dO_t . v_s) goes to dcum_t (+) and dcum_s (-). Summed
//     over a node the query side is r_{t,p} q_t^T B dO_t and the key side
//     w_s k_s^T C_i v_s (the block-end terms cancel). Finally
//     dlog_a_r = sum_{t >= r} dcum_t (bwd_dloga).
#include "lla_internal.cuh"

namespace lla {
namespace {

constexpr int kThreads = 256;
constexpr int kPieceTokens = 512;  // query tokens per block of the node-gradient kernel
constexpr int kMaxChunk = 64;      // chunk length used by the backward

struct Offsets { int off[32]; };

// Inclusive prefix sum of n <= 128 values by one warp (lane l owns 4 consecutive values).
__device__ void warp_prefix(const float* src, float* dst, int n) {
    const int lane = threadIdx.x & 31;
    float x[4];
    float run = 0.f;
#pragma unroll
    for (int e = 0; e < 4; e++) {
        const int idx = lane * 4 + e;
        run += (idx < n) ? src[idx] : 0.f;
        x[e] = run;
    }
    float incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    const float excl = incl - run;
#pragma unroll
    for (int e = 0; e < 4; e++) {
        const int idx = lane * 4 + e;
        if (idx < n) dst[idx] = x[e] + excl;
    }
}

// dB_{p,m} += sum over one piece (<= 512 tokens) of its query block of r_{t,p} q_t dO_t^T.
// grid (read nodes, pieces, BH), 256 threads as 16 x 16: thread (ty, tx) owns rows
// d = ty + 16 a (a < AD) and columns e = tx + 16 b (b < BE) of the dk x dv matrix.
template <typename T, int AD, int BE>
__global__ void __launch_bounds__(kThreads)
    bwd_dnode_kernel(const T* __restrict__ q, const T* __restrict__ dout, const float* __restrict__ log_a,
                     const float* __restrict__ lambda, const float* __restrict__ g, float* __restrict__ dnodes,
                     int Tlen, int dk, int dv, int chunk, int c, int N, int P, int L, int node_count, Offsets lo,
                     Offsets ro) {
    __shared__ float qw[32][129];
    __shared__ float go[32][129];
    __shared__ float araw[kMaxChunk], cl[kMaxChunk];
    __shared__ float e0_sh;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int idx = blockIdx.x, piece = blockIdx.y, bh = blockIdx.z;
    int p = 0;
    while (p + 1 < P && ro.off[p + 1] <= idx) p++;
    const int m = 2 * (idx - ro.off[p]);
    const int qc0 = (m + 1) << p;
    const int qc1 = min((m + 2) << p, N);
    const int tb = qc0 * chunk + piece * kPieceTokens;
    if (tb >= qc1 * chunk) return;
    const int te = min(tb + kPieceTokens, qc1 * chunk);
    const size_t row0 = static_cast<size_t>(bh) * Tlen;
    // decay exponent from the block end e = qc0 C - 1 to the token before this piece
    if (tid < 32) {
        float sacc = 0.f;
        for (int i = qc0 + tid; i < tb / chunk; i += 32) sacc += g[static_cast<size_t>(bh) * N + i];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sacc += __shfl_xor_sync(0xffffffffu, sacc, off);
        if (tid == 0) e0_sh = sacc;
    }
    __syncthreads();
    float E0 = e0_sh;
    const int lev = c + 1 + p;
    float acc[AD][BE];
#pragma unroll
    for (int a = 0; a < AD; a++)
#pragma unroll
        for (int b = 0; b < BE; b++) acc[a][b] = 0.f;
    for (int cs = tb; cs < te; cs += chunk) {
        for (int u = tid; u < chunk; u += kThreads) araw[u] = log_a[row0 + cs + u];
        __syncthreads();
        if (tid < 32) warp_prefix(araw, cl, chunk);
        __syncthreads();
        for (int st = 0; st < chunk; st += 32) {
            const int ns = min(32, chunk - st);
            for (int x = tid; x < ns * dk; x += kThreads) {
                const int sl = x / dk, d = x % dk;
                const size_t t = row0 + cs + st + sl;
                const float w = lambda[t * L + lev] * expf(E0 + cl[st + sl]);
                qw[sl][d] = w * load_f(q + t * dk + d);
            }
            for (int x = tid; x < ns * dv; x += kThreads) {
                const int sl = x / dv, e = x % dv;
                go[sl][e] = load_f(dout + (row0 + cs + st + sl) * dv + e);
            }
            __syncthreads();
            for (int sl = 0; sl < ns; sl++) {
                float av[AD], bv[BE];
#pragma unroll
                for (int a = 0; a < AD; a++) av[a] = qw[sl][ty + 16 * a];
#pragma unroll
                for (int b = 0; b < BE; b++) bv[b] = go[sl][tx + 16 * b];
#pragma unroll
                for (int a = 0; a < AD; a++)
#pragma unroll
                    for (int b = 0; b < BE; b++) acc[a][b] = fmaf(av[a], bv[b], acc[a][b]);
            }
            __syncthreads();
        }
        E0 += cl[chunk - 1];
        __syncthreads();
    }
    float* dst = dnodes + (static_cast<size_t>(bh) * node_count + lo.off[p] + m) * static_cast<size_t>(dk * dv);
#pragma unroll
    for (int a = 0; a < AD; a++)
#pragma unroll
        for (int b = 0; b < BE; b++) {
            const int d = ty + 16 * a, e = tx + 16 * b;
            if (d < dk && e < dv) atomicAdd(dst + d * dv + e, acc[a][b]);
        }
}

// Block log-decay totals of every node, same indexing as the nodes. grid (BH).
__global__ void __launch_bounds__(kThreads) bwd_blocktot_kernel(const float* __restrict__ g, float* __restrict__ gtab,
                                                                int N, int P, int node_count, Offsets lo) {
    const int bh = blockIdx.x;
    float* G = gtab + static_cast<size_t>(bh) * node_count;
    for (int m = threadIdx.x; m < N; m += kThreads) G[m] = g[static_cast<size_t>(bh) * N + m];
    __syncthreads();
    for (int p = 1; p < P; p++) {
        for (int m = threadIdx.x; m < (N >> p); m += kThreads)
            G[lo.off[p] + m] = G[lo.off[p - 1] + 2 * m] + G[lo.off[p - 1] + 2 * m + 1];
        __syncthreads();
    }
}

// One level of the top-down pass: for every node (p, m) whose parent exists,
// X_{p,m} += decay(end of (p,m) -> end of parent) X_{p+1,m>>1}, where the decay is 1
// for a right child and exp(G_{p,m+1}) for a left one. Starting from X = dB and
// running p = P-2 .. 0 leaves C_i at level 0. grid (ceil(dk*dv / 256), N >> p, BH).
__global__ void __launch_bounds__(kThreads) bwd_topdown_level_kernel(float* __restrict__ dnodes,
                                                                     const float* __restrict__ gtab, int p, int N,
                                                                     int node_count, int msz, Offsets lo) {
    const int e = blockIdx.x * kThreads + threadIdx.x;
    const int m = blockIdx.y, bh = blockIdx.z;
    const int par = m >> 1;
    if (e >= msz || par >= (N >> (p + 1))) return;
    const float* G = gtab + static_cast<size_t>(bh) * node_count;
    const float dec = (m & 1) ? 1.f : expf(G[lo.off[p] + m + 1]);
    float* base = dnodes + static_cast<size_t>(bh) * node_count * msz + e;
    base[static_cast<size_t>(lo.off[p] + m) * msz] += dec * base[static_cast<size_t>(lo.off[p + 1] + par) * msz];
}

// Everything for the tokens of one chunk j. grid (N, BH), 256 threads as 16 x 16,
// dynamic shared memory (see chunk_smem_floats).
template <typename T>
__global__ void __launch_bounds__(kThreads)
    bwd_chunk_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     const float* __restrict__ log_a, const float* __restrict__ lambda, const T* __restrict__ dout,
                     const float* __restrict__ g, const float* __restrict__ nodes, const float* __restrict__ cnodes,
                     T* __restrict__ dq, T* __restrict__ dk_out, T* __restrict__ dv_out, float* __restrict__ dlambda,
                     float* __restrict__ dcum, int Tlen, int dk, int dv, int chunk, int c, int N, int P, int L,
                     int node_count, Offsets lo) {
    extern __shared__ float sm[];
    __shared__ float dsum_sh;
    const int C = chunk, SK = dk + 1, SV = dv + 1, SC = C + 1;
    float* qs = sm;                 // [C][SK]
    float* ks = qs + C * SK;        // [C][SK]
    float* vs = ks + C * SK;        // [C][SV]
    float* gs = vs + C * SV;        // [C][SV]  dO
    float* Am = gs + C * SV;        // [C][SC]  A_ts
    float* Gm = Am + C * SC;        // [C][SC]  G_ts
    float* stg = Gm + C * SC;       // staging, 128 x 33 or 32 x 129
    float* cl = stg + 128 * 33;     // [C] in-chunk inclusive prefix of log_a
    float* araw = cl + kMaxChunk;   // [C]
    float* lam = araw + kMaxChunk;  // [C][L]
    float* dlam = lam + C * L;      // [C][L]
    float* dcs = dlam + C * L;      // [C] dcum of the chunk's tokens

    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int j = blockIdx.x, bh = blockIdx.y;
    const size_t row0 = static_cast<size_t>(bh) * Tlen + static_cast<size_t>(j) * C;
    const int NA = C / 16;  // row groups: rows ty + 16 a, a < NA

    for (int x = tid; x < C * dk; x += kThreads) {
        const int r = x / dk, d = x % dk;
        qs[r * SK + d] = load_f(q + (row0 + r) * dk + d);
        ks[r * SK + d] = load_f(k + (row0 + r) * dk + d);
    }
    for (int x = tid; x < C * dv; x += kThreads) {
        const int r = x / dv, e = x % dv;
        vs[r * SV + e] = load_f(v + (row0 + r) * dv + e);
        gs[r * SV + e] = load_f(dout + (row0 + r) * dv + e);
    }
    for (int x = tid; x < C * L; x += kThreads) {
        lam[x] = lambda[row0 * L + x];
        dlam[x] = 0.f;
    }
    for (int u = tid; u < C; u += kThreads) {
        araw[u] = log_a[row0 + u];
        dcs[u] = 0.f;
    }
    __syncthreads();
    if (tid < 32) warp_prefix(araw, cl, C);
    __syncthreads();

    // ---- pairs inside the chunk: t = ty + 16 a, s = tx + 16 b
    {
        float qk[4][4], gv[4][4];
#pragma unroll
        for (int a = 0; a < 4; a++)
#pragma unroll
            for (int b = 0; b < 4; b++) qk[a][b] = gv[a][b] = 0.f;
        for (int d = 0; d < dk; d++) {
            float qa[4], kb[4];
#pragma unroll
            for (int a = 0; a < 4; a++) qa[a] = a < NA ? qs[(ty + 16 * a) * SK + d] : 0.f;
#pragma unroll
            for (int b = 0; b < 4; b++) kb[b] = b < NA ? ks[(tx + 16 * b) * SK + d] : 0.f;
#pragma unroll
            for (int a = 0; a < 4; a++)
#pragma unroll
                for (int b = 0; b < 4; b++) qk[a][b] = fmaf(qa[a], kb[b], qk[a][b]);
        }
        for (int e = 0; e < dv; e++) {
            float ga[4], vb[4];
#pragma unroll
            for (int a = 0; a < 4; a++) ga[a] = a < NA ? gs[(ty + 16 * a) * SV + e] : 0.f;
#pragma unroll
            for (int b = 0; b < 4; b++) vb[b] = b < NA ? vs[(tx + 16 * b) * SV + e] : 0.f;
#pragma unroll
            for (int a = 0; a < 4; a++)
#pragma unroll
                for (int b = 0; b < 4; b++) gv[a][b] = fmaf(ga[a], vb[b], gv[a][b]);
        }
#pragma unroll
        for (int a = 0; a < 4; a++) {
            if (a >= NA) break;
            const int t = ty + 16 * a;
            float erow = 0.f;
#pragma unroll
            for (int b = 0; b < 4; b++) {
                if (b >= NA) break;
                const int s = tx + 16 * b;
                float A = 0.f, Gv = 0.f;
                if (s <= t) {
                    const int l = fenwick_level(t, s);  // same high bits: local positions suffice
                    const float D = expf(cl[t] - cl[s]);
                    const float lm = lam[t * L + l];
                    const float dqkgv = D * qk[a][b] * gv[a][b];
                    A = lm * D * qk[a][b];
                    Gv = lm * D * gv[a][b];
                    atomicAdd(&dlam[t * L + l], dqkgv);
                    const float E = lm * dqkgv;
                    erow += E;
                    atomicAdd(&dcs[s], -E);
                }
                Am[t * SC + s] = A;
                Gm[t * SC + s] = Gv;
            }
            atomicAdd(&dcs[t], erow);
        }
    }
    __syncthreads();

    const float* cj = (P > 0) ? cnodes + (static_cast<size_t>(bh) * node_count + lo.off[0] + j) * (size_t)(dk * dv)
                              : nullptr;
    const int NB_K = (dk + 15) / 16, NB_V = (dv + 15) / 16;

    // ---- dq: rows t, columns d
    {
        float acc[4][8];
#pragma unroll
        for (int a = 0; a < 4; a++)
#pragma unroll
            for (int b = 0; b < 8; b++) acc[a][b] = 0.f;
        for (int s = 0; s < C; s++) {
            float ga[4], kb[8];
#pragma unroll
            for (int a = 0; a < 4; a++) ga[a] = a < NA ? Gm[(ty + 16 * a) * SC + s] : 0.f;
#pragma unroll
            for (int b = 0; b < 8; b++) kb[b] = (b < NB_K && tx + 16 * b < dk) ? ks[s * SK + tx + 16 * b] : 0.f;
#pragma unroll
            for (int a = 0; a < 4; a++)
#pragma unroll
                for (int b = 0; b < 8; b++) acc[a][b] = fmaf(ga[a], kb[b], acc[a][b]);
        }
        // Fenwick node reads: B dO_t for every set bit p of j
        for (int p = 0; p < P; p++) {
            if (((j >> p) & 1) == 0) continue;
            const int m = (j >> p) - 1;
            __syncthreads();  // every thread has read the previous level's dsum_sh
            if (tid < 32) {
                float d_ = 0.f;
                for (int i = ((j >> p) << p) + tid; i < j; i += 32) d_ += g[static_cast<size_t>(bh) * N + i];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) d_ += __shfl_xor_sync(0xffffffffu, d_, off);
                if (tid == 0) dsum_sh = d_;
            }
            const float* node = nodes + (static_cast<size_t>(bh) * node_count + lo.off[p] + m) * (size_t)(dk * dv);
            float tmp[4][8];
#pragma unroll
            for (int a = 0; a < 4; a++)
#pragma unroll
                for (int b = 0; b < 8; b++) tmp[a][b] = 0.f;
            for (int e0 = 0; e0 < dv; e0 += 32) {
                const int ne = min(32, dv - e0);
                __syncthreads();
                for (int x = tid; x < dk * 32; x += kThreads) {
                    const int d = x >> 5, ee = x & 31;
                    stg[d * 33 + ee] = ee < ne ? node[static_cast<size_t>(d) * dv + e0 + ee] : 0.f;
                }
                __syncthreads();
                for (int ee = 0; ee < ne; ee++) {
                    float ga[4], bb[8];
#pragma unroll
                    for (int a = 0; a < 4; a++) ga[a] = a < NA ? gs[(ty + 16 * a) * SV + e0 + ee] : 0.f;
#pragma unroll
                    for (int b = 0; b < 8; b++) bb[b] = (b < NB_K && tx + 16 * b < dk) ? stg[(tx + 16 * b) * 33 + ee] : 0.f;
#pragma unroll
                    for (int a = 0; a < 4; a++)
#pragma unroll
                        for (int b = 0; b < 8; b++) tmp[a][b] = fmaf(ga[a], bb[b], tmp[a][b]);
                }
            }
            const float dsum = dsum_sh;
#pragma unroll
            for (int a = 0; a < 4; a++) {
                if (a >= NA) break;
                const int t = ty + 16 * a;
                const float rho = expf(cl[t] + dsum);
                const float r = lam[t * L + c + 1 + p] * rho;
                float z = 0.f;
#pragma unroll
                for (int b = 0; b < 8; b++) {
                    const int d = tx + 16 * b;
                    if (b < NB_K && d < dk) z = fmaf(qs[t * SK + d], tmp[a][b], z);
                    acc[a][b] = fmaf(r, tmp[a][b], acc[a][b]);
                }
#pragma unroll
                for (int off = 1; off < 16; off <<= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
                if (tx == 0) {
                    dlam[t * L + c + 1 + p] = rho * z;
                    dcs[t] += r * z;
                }
            }
        }
#pragma unroll
        for (int a = 0; a < 4; a++) {
            if (a >= NA) break;
            const int t = ty + 16 * a;
#pragma unroll
            for (int b = 0; b < 8; b++) {
                const int d = tx + 16 * b;
                if (b < NB_K && d < dk) store_f(dq + (row0 + t) * dk + d, acc[a][b]);
            }
        }
    }
    __syncthreads();

    // ---- dk: rows s, columns d
    {
        float acc[4][8];
#pragma unroll
        for (int a = 0; a < 4; a++)
#pragma unroll
            for (int b = 0; b < 8; b++) acc[a][b] = 0.f;
        for (int t = 0; t < C; t++) {
            float ga[4], qb[8];
#pragma unroll
            for (int a = 0; a < 4; a++) ga[a] = a < NA ? Gm[t * SC + ty + 16 * a] : 0.f;
#pragma unroll
            for (int b = 0; b < 8; b++) qb[b] = (b < NB_K && tx + 16 * b < dk) ? qs[t * SK + tx + 16 * b] : 0.f;
#pragma unroll
            for (int a = 0; a < 4; a++)
#pragma unroll
                for (int b = 0; b < 8; b++) acc[a][b] = fmaf(ga[a], qb[b], acc[a][b]);
        }
        if (cj) {
            float tmp[4][8];
#pragma unroll
            for (int a = 0; a < 4; a++)
#pragma unroll
                for (int b = 0; b < 8; b++) tmp[a][b] = 0.f;
            for (int e0 = 0; e0 < dv; e0 += 32) {
                const int ne = min(32, dv - e0);
                __syncthreads();
                for (int x = tid; x < dk * 32; x += kThreads) {
                    const int d = x >> 5, ee = x & 31;
                    stg[d * 33 + ee] = ee < ne ? cj[static_cast<size_t>(d) * dv + e0 + ee] : 0.f;
                }
                __syncthreads();
                for (int ee = 0; ee < ne; ee++) {
                    float va[4], cb[8];
#pragma unroll
                    for (int a = 0; a < 4; a++) va[a] = a < NA ? vs[(ty + 16 * a) * SV + e0 + ee] : 0.f;
#pragma unroll
                    for (int b = 0; b < 8; b++) cb[b] = (b < NB_K && tx + 16 * b < dk) ? stg[(tx + 16 * b) * 33 + ee] : 0.f;
#pragma unroll
                    for (int a = 0; a < 4; a++)
#pragma unroll
                        for (int b = 0; b < 8; b++) tmp[a][b] = fmaf(va[a], cb[b], tmp[a][b]);
                }
            }
#pragma unroll
            for (int a = 0; a < 4; a++) {
                if (a >= NA) break;
                const int s = ty + 16 * a;
                const float w = expf(cl[C - 1] - cl[s]);
                float y = 0.f;
#pragma unroll
                for (int b = 0; b < 8; b++) {
                    const int d = tx + 16 * b;
                    if (b < NB_K && d < dk) y = fmaf(ks[s * SK + d], tmp[a][b], y);
                    acc[a][b] = fmaf(w, tmp[a][b], acc[a][b]);
                }
#pragma unroll
                for (int off = 1; off < 16; off <<= 1) y += __shfl_xor_sync(0xffffffffu, y, off);
                if (tx == 0) dcs[s] -= w * y;
            }
        }
#pragma unroll
        for (int a = 0; a < 4; a++) {
            if (a >= NA) break;
            const int s = ty + 16 * a;
#pragma unroll
            for (int b = 0; b < 8; b++) {
                const int d = tx + 16 * b;
                if (b < NB_K && d < dk) store_f(dk_out + (row0 + s) * dk + d, acc[a][b]);
            }
        }
    }
    __syncthreads();

    // ---- dv: rows s, columns e
    {
        float acc[4][8];
#pragma unroll
        for (int a = 0; a < 4; a++)
#pragma unroll
            for (int b = 0; b < 8; b++) acc[a][b] = 0.f;
        for (int t = 0; t < C; t++) {
            float aa[4], gb[8];
#pragma unroll
            for (int a = 0; a < 4; a++) aa[a] = a < NA ? Am[t * SC + ty + 16 * a] : 0.f;
#pragma unroll
            for (int b = 0; b < 8; b++) gb[b] = (b < NB_V && tx + 16 * b < dv) ? gs[t * SV + tx + 16 * b] : 0.f;
#pragma unroll
            for (int a = 0; a < 4; a++)
#pragma unroll
                for (int b = 0; b < 8; b++) acc[a][b] = fmaf(aa[a], gb[b], acc[a][b]);
        }
        if (cj) {
            float tmp[4][8];
#pragma unroll
            for (int a = 0; a < 4; a++)
#pragma unroll
                for (int b = 0; b < 8; b++) tmp[a][b] = 0.f;
            for (int d0 = 0; d0 < dk; d0 += 32) {
                const int nd = min(32, dk - d0);
                __syncthreads();
                for (int x = tid; x < 32 * dv; x += kThreads) {
                    const int dd = x / dv, e = x % dv;
                    stg[dd * 129 + e] = dd < nd ? cj[static_cast<size_t>(d0 + dd) * dv + e] : 0.f;
                }
                __syncthreads();
                for (int dd = 0; dd < nd; dd++) {
                    float ka[4], cb[8];
#pragma unroll
                    for (int a = 0; a < 4; a++) ka[a] = a < NA ? ks[(ty + 16 * a) * SK + d0 + dd] : 0.f;
#pragma unroll
                    for (int b = 0; b < 8; b++) cb[b] = (b < NB_V && tx + 16 * b < dv) ? stg[dd * 129 + tx + 16 * b] : 0.f;
#pragma unroll
                    for (int a = 0; a < 4; a++)
#pragma unroll
                        for (int b = 0; b < 8; b++) tmp[a][b] = fmaf(ka[a], cb[b], tmp[a][b]);
                }
            }
#pragma unroll
            for (int a = 0; a < 4; a++) {
                if (a >= NA) break;
                const float w = expf(cl[C - 1] - cl[ty + 16 * a]);
#pragma unroll
                for (int b = 0; b < 8; b++) acc[a][b] = fmaf(w, tmp[a][b], acc[a][b]);
            }
        }
#pragma unroll
        for (int a = 0; a < 4; a++) {
            if (a >= NA) break;
            const int s = ty + 16 * a;
#pragma unroll
            for (int b = 0; b < 8; b++) {
                const int e = tx + 16 * b;
                if (b < NB_V && e < dv) store_f(dv_out + (row0 + s) * dv + e, acc[a][b]);
            }
        }
    }
    __syncthreads();
    for (int x = tid; x < C * L; x += kThreads) dlambda[row0 * L + x] = dlam[x];
    for (int u = tid; u < C; u += kThreads) dcum[row0 + u] = dcs[u];
}

size_t chunk_smem_floats(int C, int dk, int dv, int L) {
    return static_cast<size_t>(C) * (2 * (dk + 1) + 2 * (dv + 1) + 2 * (C + 1) + 2 * L) + 128 * 33 + 3 * kMaxChunk;
}

// dlog_a_r = sum_{t >= r} dcum_t, per head. grid (BH), 1024 threads. The head is taken in
// pieces of 8192 tokens from its end: a coalesced copy into shared memory, suffix sums over
// 8 consecutive tokens per thread, a block-wide suffix scan of those sums, a coalesced store.
constexpr int kDlogaThreads = 1024;
constexpr int kDlogaPiece = 8 * kDlogaThreads;

__global__ void __launch_bounds__(kDlogaThreads) bwd_dloga_kernel(const float* __restrict__ dcum,
                                                                 float* __restrict__ dlog_a, int Tlen) {
    __shared__ float buf[kDlogaPiece];
    __shared__ float warp_tot[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float* src = dcum + static_cast<size_t>(blockIdx.x) * Tlen;
    float* dst = dlog_a + static_cast<size_t>(blockIdx.x) * Tlen;
    float carry = 0.f;  // sum of the tokens after this piece
    for (int end = Tlen; end > 0; end -= kDlogaPiece) {
        const int beg = end > kDlogaPiece ? end - kDlogaPiece : 0, n = end - beg;
        for (int i = tid; i < n; i += kDlogaThreads) buf[i] = src[beg + i];
        __syncthreads();
        float v[8], tot = 0.f;
#pragma unroll
        for (int e = 7; e >= 0; e--) {
            const int i = 8 * tid + e;
            tot += i < n ? buf[i] : 0.f;
            v[e] = tot;
        }
        // suffix scan of the thread totals: lanes after this one, then warps after this one
        float incl = tot;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_down_sync(0xffffffffu, incl, off);
            if (lane + off < 32) incl += y;
        }
        if (lane == 0) warp_tot[warp] = incl;
        __syncthreads();
        float after = carry + incl - tot;
        for (int w = warp + 1; w < 32; w++) after += warp_tot[w];
#pragma unroll
        for (int e = 0; e < 8; e++) {
            const int i = 8 * tid + e;
            if (i < n) buf[i] = v[e] + after;
        }
        float piece = 0.f;
        for (int w = 0; w < 32; w++) piece += warp_tot[w];
        __syncthreads();
        for (int i = tid; i < n; i += kDlogaThreads) dst[beg + i] = buf[i];
        carry += piece;
        __syncthreads();
    }
}

template <typename T>
cudaError_t backward_t(const BwdPlan& pl, const T* q, const T* k, const T* v, const float* log_a,
                       const float* lambda, const T* dout, T* dq, T* dk, T* dv, float* dlog_a, float* dlambda,
                       void* workspace, cudaStream_t stream) {
    const SimtPlan& fw = pl.fw;
    const int BH = fw.B * fw.H;
    const int L = bitlength(static_cast<int64_t>(fw.T) - 1) + 1;
    const int msz = fw.dk * fw.dv;
    char* ws = static_cast<char*>(workspace);
    const float* g = reinterpret_cast<const float*>(ws);
    const float* nodes = reinterpret_cast<const float*>(ws + fw.g_bytes);
    float* dnodes = reinterpret_cast<float*>(ws + fw.total_bytes);
    float* gtab = reinterpret_cast<float*>(ws + fw.total_bytes + pl.dnodes_bytes);
    float* dcum = reinterpret_cast<float*>(ws + fw.total_bytes + pl.dnodes_bytes +
                                           ((static_cast<size_t>(BH) * fw.node_count * sizeof(float) + 255) / 256 * 256));
    Offsets lo, ro;
    for (int p = 0; p < 32; p++) {
        lo.off[p] = fw.level_off[p];
        ro.off[p] = pl.read_off[p];
    }
    cudaError_t e = simt_nodes(fw, sizeof(T) == 4 ? 1 : 0, k, v, log_a, workspace, stream);
    if (e != cudaSuccess) return e;
    note_launch(stream, "simt_nodes");
    if (fw.node_count > 0) {
        e = cudaMemsetAsync(dnodes, 0, pl.dnodes_bytes, stream);
        if (e != cudaSuccess) return e;
    }
    if (pl.n_read > 0) {
        const dim3 grid(pl.n_read, pl.max_pieces, BH);
        const bool wk = fw.dk > 64, wv = fw.dv > 64;
        if (wk && wv)
            bwd_dnode_kernel<T, 8, 8><<<grid, kThreads, 0, stream>>>(q, dout, log_a, lambda, g, dnodes, fw.T, fw.dk,
                                                                     fw.dv, fw.chunk, fw.c, fw.N, fw.P, L,
                                                                     fw.node_count, lo, ro);
        else if (wk)
            bwd_dnode_kernel<T, 8, 4><<<grid, kThreads, 0, stream>>>(q, dout, log_a, lambda, g, dnodes, fw.T, fw.dk,
                                                                     fw.dv, fw.chunk, fw.c, fw.N, fw.P, L,
                                                                     fw.node_count, lo, ro);
        else if (wv)
            bwd_dnode_kernel<T, 4, 8><<<grid, kThreads, 0, stream>>>(q, dout, log_a, lambda, g, dnodes, fw.T, fw.dk,
                                                                     fw.dv, fw.chunk, fw.c, fw.N, fw.P, L,
                                                                     fw.node_count, lo, ro);
        else
            bwd_dnode_kernel<T, 4, 4><<<grid, kThreads, 0, stream>>>(q, dout, log_a, lambda, g, dnodes, fw.T, fw.dk,
                                                                     fw.dv, fw.chunk, fw.c, fw.N, fw.P, L,
                                                                     fw.node_count, lo, ro);
        note_launch(stream, "bwd_dnode");
    }
    if (fw.P > 1) {
        bwd_blocktot_kernel<<<BH, kThreads, 0, stream>>>(g, gtab, fw.N, fw.P, fw.node_count, lo);
        for (int p = fw.P - 2; p >= 0; p--)
            bwd_topdown_level_kernel<<<dim3((msz + kThreads - 1) / kThreads, fw.N >> p, BH), kThreads, 0, stream>>>(
                dnodes, gtab, p, fw.N, fw.node_count, msz, lo);
        note_launch(stream, "bwd_topdown");
    }
    {
        const size_t smem = chunk_smem_floats(fw.chunk, fw.dk, fw.dv, L) * sizeof(float);
        e = cudaFuncSetAttribute(bwd_chunk_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        bwd_chunk_kernel<T><<<dim3(fw.N, BH), kThreads, smem, stream>>>(
            q, k, v, log_a, lambda, dout, g, nodes, dnodes, dq, dk, dv, dlambda, dcum, fw.T, fw.dk, fw.dv, fw.chunk,
            fw.c, fw.N, fw.P, L, fw.node_count, lo);
        note_launch(stream, "bwd_chunk");
    }
    bwd_dloga_kernel<<<BH, kDlogaThreads, 0, stream>>>(dcum, dlog_a, fw.T);
    note_launch(stream, "bwd_dloga");
    return cudaGetLastError();
}

}  // namespace

cudaError_t bwd_dloga(const float* dcum, float* dlog_a, int BH, int T, cudaStream_t stream) {
    bwd_dloga_kernel<<<BH, kDlogaThreads, 0, stream>>>(dcum, dlog_a, T);
    note_launch(stream, "bwd_dloga");
    return cudaGetLastError();
}

bool make_bwd_plan(int B, int H, int T, int dk, int dv, int chunk, BwdPlan* pl) {
    const int C = chunk < kMaxChunk ? chunk : kMaxChunk;
    if (T % C != 0) return false;
    const int L = bitlength(static_cast<int64_t>(T) - 1) + 1;
    if (L > 32) return false;
    if (chunk_smem_floats(C, dk, dv, L) * sizeof(float) > 227 * 1024) return false;
    if (!make_simt_plan(B, H, T, dk, dv, C, &pl->fw)) return false;
    const SimtPlan& fw = pl->fw;
    int n = 0;
    for (int p = 0; p < 32; p++) {
        pl->read_off[p] = n;
        if (p < fw.P) n += (((fw.N - 1) >> p) + 1) / 2;  // even m with (m + 1) 2^p < N
    }
    pl->n_read = n;
    const int64_t big_block = fw.P > 0 ? (static_cast<int64_t>(1) << (fw.P - 1)) * C : 0;
    pl->max_pieces = static_cast<int>((big_block + kPieceTokens - 1) / kPieceTokens);
    if (pl->max_pieces < 1) pl->max_pieces = 1;
    if (pl->max_pieces > 65535) return false;
    const size_t BH = static_cast<size_t>(B) * H;
    pl->dnodes_bytes = (BH * fw.node_count * static_cast<size_t>(dk) * dv * sizeof(float) + 255) / 256 * 256;
    const size_t gtab_bytes = (BH * fw.node_count * sizeof(float) + 255) / 256 * 256;
    pl->dcum_bytes = (BH * static_cast<size_t>(T) * sizeof(float) + 255) / 256 * 256;
    pl->total_bytes = fw.total_bytes + pl->dnodes_bytes + gtab_bytes + pl->dcum_bytes;
    return true;
}

cudaError_t simt_backward(const BwdPlan& pl, int dtype, const void* q, const void* k, const void* v,
                          const float* log_a, const float* lambda, const void* dout, void* dq, void* dk, void* dv,
                          float* dlog_a, float* dlambda, void* workspace, cudaStream_t stream) {
    if (dtype == 1)
        return backward_t<float>(pl, static_cast<const float*>(q), static_cast<const float*>(k),
                                 static_cast<const float*>(v), log_a, lambda, static_cast<const float*>(dout),
                                 static_cast<float*>(dq), static_cast<float*>(dk), static_cast<float*>(dv), dlog_a,
                                 dlambda, workspace, stream);
    using B16 = __nv_bfloat16;
    return backward_t<B16>(pl, static_cast<const B16*>(q), static_cast<const B16*>(k), static_cast<const B16*>(v),
                           log_a, lambda, static_cast<const B16*>(dout), static_cast<B16*>(dq),
                           static_cast<B16*>(dk), static_cast<B16*>(dv), dlog_a, dlambda, workspace, stream);
}

}  // namespace lla
