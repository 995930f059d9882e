// Log-linear Gated DeltaNet ("Log-Linear Attention", pt §2 "Generalizacao" and
// fr §3 "Etudes de Cas": the hierarchical mask applied to Gated DeltaNet).
//
//   o_t = sum_{s<=t} lambda_t^(l(t,s)) A[t,s] v_s,
//   A[t,s] = beta_s k_s^T A_{s+1} ... A_t q_t,   A_r = alpha_r (I - beta_r k_r k_r^T),
//
// alpha_r = exp(log_a_r). Recurrently every held Fenwick bucket state S (dk x dv)
// evolves as S <- A_t S, buckets merge on the lowbit carry and the new token writes
// beta_t k_t v_t^T at level 0 (pt §2 "Forma Recorrente e Paralela").
//
// Decode: one CTA per (b, h); each held level is read once and written once.
// Per level the two column reductions w = k^T S and z = q^T S give both the update
// S' = alpha (S - beta k w^T) and the level's output lambda alpha (z - beta (q.k) w).
//
// Prefill (chunkwise: dense work inside a chunk of C tokens, hierarchical state
// passing between chunks, fr §2 "Algorithmes Efficaces"). Scalars commute with the
// transitions, so a product of them is a decay times a product of (I - beta k k^T).
// Per chunk (gdn_chunk_kernel), with cl the in-chunk prefix of log a:
//   Lk = (I + diag(beta) strictlower(K K^T))^-1 and W = Lk diag(beta) K: the chunk's
//        transition product A_{first} ... A_t = e^{cl_t} (I - sum_{r<=t} w_r k_r^T);
//   Q~ = diag(e^{cl}) (Q - tril(Q K^T) W): row t is A_{first} ... A_t q_t, the query
//        carried back to the chunk start, so a state X held at the chunk start is
//        read as X^T q~_t;
//   Lg = (I + diag(beta) (Gamma (.) strictlower(K K^T)))^-1, Gamma_ts = e^{cl_t - cl_s}:
//        the delta rule's pseudo-values U = Lg diag(beta) V, the chunk's own state
//        S = K^T diag(e^{cl_end - cl}) U (the level-0 node), and its attention matrix
//        A = tril(Gamma (.) Q K^T) Lg diag(beta), read with lambda^(l(t,s)) inside the chunk.
// Per Fenwick level p (gdn_level_kernel, one launch per level, levels in order):
// node (p, m) holds the state of chunks [m 2^p, (m+1) 2^p) at its end; for m even it
// is carried forward chunk by chunk through the next block (X <- gamma_j (X - K_j^T (W_j X))),
// read at each chunk j there with lambda^(c+1+p) X^T q~_t, and the carried node plus
// node (p, m+1) is node (p+1, m/2).
// Every kernel computes in fp32 on CUDA cores.
#include "lla_internal.cuh"

namespace lla {
namespace {

constexpr int kGdnThreads = 256;

struct GdnLevels { int off[32]; };  // first node of each level in a head's node array

// ------------------------------------------------------------------ decode

template <typename T, int DV4, int DK>
__global__ void __launch_bounds__(256) gdn_decode_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                         const T* __restrict__ v, const float* __restrict__ log_a,
                                                         const float* __restrict__ beta,
                                                         const float* __restrict__ lambda,
                                                         float* __restrict__ states, const int64_t* __restrict__ tpos,
                                                         T* __restrict__ out, int H, int Lmax, int* err) {
    constexpr int DV = DV4 * 4;
    constexpr int RPT = DK * DV4 / 256 > 1 ? DK * DV4 / 256 : 1;  // rows per thread
    constexpr int NTH = DV4 * DK / RPT;                            // threads launched
    constexpr int RPP = NTH / DV4;                                 // rows per pass
    constexpr int NW = NTH / 32;
    static_assert(NTH % 32 == 0 && NTH <= 256, "thread count");
    __shared__ float qsh[DK], ksh[DK];
    __shared__ float vsh[DV];
    __shared__ float lam[40];
    __shared__ float4 red[2][NW][DV4];
    __shared__ float qk_sh;
    const int tid = threadIdx.x;
    const int bh = blockIdx.x;
    const int b = bh / H;
    const int64_t tb = tpos[b];
    if (tb < 0 || tb >= ((int64_t)1 << (Lmax - 1))) {
        if (tid == 0) record_error(err, kDevBadInput);
        return;
    }
    for (int x = tid; x < DK; x += NTH) {
        qsh[x] = load_f(q + (size_t)bh * DK + x);
        ksh[x] = load_f(k + (size_t)bh * DK + x);
    }
    for (int x = tid; x < DV; x += NTH) vsh[x] = load_f(v + (size_t)bh * DV + x);
    for (int x = tid; x < Lmax; x += NTH) lam[x] = lambda[(size_t)bh * Lmax + x];
    __syncthreads();
    if (tid < 32) {
        float s = 0.f;
        for (int x = tid; x < DK; x += 32) s += qsh[x] * ksh[x];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (tid == 0) qk_sh = s;
    }
    __syncthreads();
    const float alpha = expf(log_a[bh]);
    const float bt = beta[bh];
    const float qk = qk_sh;
    const int col4 = tid % DV4;
    const int row0 = tid / DV4;
    const int warp = tid >> 5, lane = tid & 31;
    constexpr size_t msz4 = (size_t)DK * DV4;
    float4* S = reinterpret_cast<float4*>(states) + (size_t)bh * Lmax * msz4 + (size_t)row0 * DV4 + col4;
    constexpr size_t rstep = (size_t)RPP * DV4;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);

    // S <- alpha (S - beta k (k^T S)) for one level held in x, stored to level `dst`;
    // adds the level's output lam_l alpha (q^T S - beta (q.k) k^T S) (one thread per columns)
    auto transit = [&](float4* x, float lam_l, int dst) {
        float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < RPT; r++) {
            const int i = row0 + r * RPP;
            const float ki = ksh[i], qi = qsh[i];
            pk.x += ki * x[r].x; pk.y += ki * x[r].y; pk.z += ki * x[r].z; pk.w += ki * x[r].w;
            pq.x += qi * x[r].x; pq.y += qi * x[r].y; pq.z += qi * x[r].z; pq.w += qi * x[r].w;
        }
#pragma unroll
        for (int off = DV4; off < 32; off <<= 1) {
            pk.x += __shfl_xor_sync(0xffffffffu, pk.x, off);
            pk.y += __shfl_xor_sync(0xffffffffu, pk.y, off);
            pk.z += __shfl_xor_sync(0xffffffffu, pk.z, off);
            pk.w += __shfl_xor_sync(0xffffffffu, pk.w, off);
            pq.x += __shfl_xor_sync(0xffffffffu, pq.x, off);
            pq.y += __shfl_xor_sync(0xffffffffu, pq.y, off);
            pq.z += __shfl_xor_sync(0xffffffffu, pq.z, off);
            pq.w += __shfl_xor_sync(0xffffffffu, pq.w, off);
        }
        if (lane < DV4) {
            red[0][warp][lane] = pk;
            red[1][warp][lane] = pq;
        }
        __syncthreads();
        float4 w = make_float4(0.f, 0.f, 0.f, 0.f), z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int ww = 0; ww < NW; ww++) {
            const float4 a4 = red[0][ww][col4], b4 = red[1][ww][col4];
            w.x += a4.x; w.y += a4.y; w.z += a4.z; w.w += a4.w;
            z.x += b4.x; z.y += b4.y; z.z += b4.z; z.w += b4.w;
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < RPT; r++) {
            const float bk = bt * ksh[row0 + r * RPP];
            float4 y;
            y.x = alpha * (x[r].x - bk * w.x);
            y.y = alpha * (x[r].y - bk * w.y);
            y.z = alpha * (x[r].z - bk * w.z);
            y.w = alpha * (x[r].w - bk * w.w);
            __stcs(S + dst * msz4 + r * rstep, y);
        }
        if (row0 == 0) {
            const float f = lam_l * alpha, g = bt * qk;
            o.x += f * (z.x - g * w.x);
            o.y += f * (z.y - g * w.y);
            o.z += f * (z.z - g * w.z);
            o.w += f * (z.w - g * w.w);
        }
    };

    if (tb > 0) {
        const int c = __ffsll((long long)tb) - 1;   // trailing zeros of t
        const int top = 64 - __clzll((long long)tb);  // bitlength(t): highest nonempty level
        // levels 0..c (all held for t-1) merge into level c+1, then take the transition
        float4 x[RPT];
#pragma unroll
        for (int r = 0; r < RPT; r++) x[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int l = 0; l <= c; l++) {
#pragma unroll
            for (int r = 0; r < RPT; r++) {
                const float4 y = __ldcs(S + l * msz4 + r * rstep);
                x[r].x += y.x; x[r].y += y.y; x[r].z += y.z; x[r].w += y.w;
            }
        }
        transit(x, lam[c + 1], c + 1);
        // coarser levels held for both t-1 and t
        for (int l = c + 2; l <= top; l++) {
            if (((tb >> (l - 1)) & 1) == 0) continue;
#pragma unroll
            for (int r = 0; r < RPT; r++) x[r] = __ldcs(S + l * msz4 + r * rstep);
            transit(x, lam[l], l);
        }
    }
    // level 0: beta_t k_t v_t^T
    {
        const float4 v4 = make_float4(vsh[col4 * 4], vsh[col4 * 4 + 1], vsh[col4 * 4 + 2], vsh[col4 * 4 + 3]);
#pragma unroll
        for (int r = 0; r < RPT; r++) {
            const float bk = bt * ksh[row0 + r * RPP];
            __stcs(S + r * rstep, make_float4(bk * v4.x, bk * v4.y, bk * v4.z, bk * v4.w));
        }
        if (row0 == 0) {
            const float f = lam[0] * bt * qk;
            o.x += f * v4.x; o.y += f * v4.y; o.z += f * v4.z; o.w += f * v4.w;
        }
    }
    if (row0 == 0) {
        T* dst = out + (size_t)bh * DV + col4 * 4;
        store_f(dst, o.x);
        store_f(dst + 1, o.y);
        store_f(dst + 2, o.z);
        store_f(dst + 3, o.w);
    }
}

template <typename T, int DV4, int DK>
cudaError_t launch_gdn_decode(const void* q, const void* k, const void* v, const float* log_a, const float* beta,
                              const float* lambda, float* states, const int64_t* t, void* out, int B, int H, int Lmax,
                              int* err, cudaStream_t stream) {
    constexpr int RPT = DK * DV4 / 256 > 1 ? DK * DV4 / 256 : 1;
    constexpr int NTH = DV4 * DK / RPT;
    gdn_decode_kernel<T, DV4, DK><<<B * H, NTH, 0, stream>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), log_a, beta, lambda, states, t,
        static_cast<T*>(out), H, Lmax, err);
    return cudaGetLastError();
}

template <typename T, int DK>
cudaError_t gdn_decode_dk(int dv, const void* q, const void* k, const void* v, const float* log_a, const float* beta,
                          const float* lambda, float* states, const int64_t* t, void* out, int B, int H, int Lmax,
                          int* err, cudaStream_t stream) {
    switch (dv) {
        case 16: return launch_gdn_decode<T, 4, DK>(q, k, v, log_a, beta, lambda, states, t, out, B, H, Lmax, err, stream);
        case 32: return launch_gdn_decode<T, 8, DK>(q, k, v, log_a, beta, lambda, states, t, out, B, H, Lmax, err, stream);
        case 64: return launch_gdn_decode<T, 16, DK>(q, k, v, log_a, beta, lambda, states, t, out, B, H, Lmax, err, stream);
        default: return launch_gdn_decode<T, 32, DK>(q, k, v, log_a, beta, lambda, states, t, out, B, H, Lmax, err, stream);
    }
}

template <typename T>
cudaError_t gdn_decode_t(int dk, int dv, const void* q, const void* k, const void* v, const float* log_a,
                         const float* beta, const float* lambda, float* states, const int64_t* t, void* out, int B,
                         int H, int Lmax, int* err, cudaStream_t stream) {
    switch (dk) {
        case 16: return gdn_decode_dk<T, 16>(dv, q, k, v, log_a, beta, lambda, states, t, out, B, H, Lmax, err, stream);
        case 32: return gdn_decode_dk<T, 32>(dv, q, k, v, log_a, beta, lambda, states, t, out, B, H, Lmax, err, stream);
        case 64: return gdn_decode_dk<T, 64>(dv, q, k, v, log_a, beta, lambda, states, t, out, B, H, Lmax, err, stream);
        default: return gdn_decode_dk<T, 128>(dv, q, k, v, log_a, beta, lambda, states, t, out, B, H, Lmax, err, stream);
    }
}

// ------------------------------------------------------------------ prefill: one chunk

constexpr int kGdnChunkThreads = 512;

// Shared-memory layout of gdn_chunk_kernel (fp32): Q, K [C][dk + 1] (rows padded so that a
// warp reading one element of 32 different rows meets 32 different banks); V [C][dv];
// W/U [C][max(dk, dv)]; G = K K^T, Gg = Gamma (.) G, QK = Q K^T (later Gamma (.) Q K^T),
// Lk, Lg [C][C]; cl, beta, the decays to the chunk end [C].
struct GdnChunkSmem {
    int C, dk, dv, ldk, wcols;
    size_t q, k, v, w, g, gg, qk, lk, lg, cl, bt, ce, total;
    __host__ __device__ GdnChunkSmem(int C_, int dk_, int dv_) : C(C_), dk(dk_), dv(dv_) {
        ldk = dk + 1;
        wcols = dk > dv ? dk : dv;
        q = 0;
        k = q + (size_t)C * ldk;
        v = k + (size_t)C * ldk;
        w = v + (size_t)C * dv;
        g = w + (size_t)C * wcols;
        gg = g + (size_t)C * C;
        qk = gg + (size_t)C * C;
        lk = qk + (size_t)C * C;
        lg = lk + (size_t)C * C;
        cl = lg + (size_t)C * C;
        bt = cl + C;
        ce = bt + C;
        total = (ce + C) * sizeof(float);
    }
};

// grid (N, BH), 512 threads; see the file header. Writes, per chunk: W and Q~ (fp32
// [BH][N][C][dk]), the chunk state (fp32 [BH][node][dk][dv], level 0 of the node
// pyramid), the chunk's total decay gamma (fp32 [BH][N]), and its in-chunk output
// (fp32 accumulator [BH][T][dv], or straight to `out` when the sequence is one chunk).
template <typename T>
__global__ void __launch_bounds__(kGdnChunkThreads) gdn_chunk_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, const float* __restrict__ log_a,
    const float* __restrict__ beta, const float* __restrict__ lambda, float* __restrict__ Wg, float* __restrict__ Qt,
    float* __restrict__ nodes, float* __restrict__ gam, float* __restrict__ oacc, T* __restrict__ out, int T_, int C,
    int dk, int dv, int L, int node_count) {
    constexpr int NT = kGdnChunkThreads;
    extern __shared__ float sm[];
    const GdnChunkSmem lay(C, dk, dv);
    const int ldk = lay.ldk, ldw = lay.wcols;
    float* Qs = sm + lay.q;
    float* Ks = sm + lay.k;
    float* Vs = sm + lay.v;
    float* Ws = sm + lay.w;
    float* G = sm + lay.g;
    float* Gg = sm + lay.gg;
    float* QK = sm + lay.qk;
    float* Lk = sm + lay.lk;
    float* Lg = sm + lay.lg;
    float* cl = sm + lay.cl;
    float* bt = sm + lay.bt;
    float* ce = sm + lay.ce;
    const int tid = threadIdx.x;
    const int j = blockIdx.x, bh = blockIdx.y;
    const int N = T_ / C;
    const size_t row0 = (size_t)bh * T_ + (size_t)j * C;

    for (int x = tid; x < C * dk; x += NT) {
        const int t = x / dk, i = x % dk;
        Qs[t * ldk + i] = load_f(q + row0 * dk + x);
        Ks[t * ldk + i] = load_f(k + row0 * dk + x);
    }
    for (int x = tid; x < C * dv; x += NT) Vs[x] = load_f(v + row0 * dv + x);
    if (tid < C) bt[tid] = beta[row0 + tid];
    if (tid < 32) {
        // in-chunk inclusive prefix of log a, 32 lanes over C <= 64 tokens
        float carry = 0.f;
        for (int base = 0; base < C; base += 32) {
            float x = base + tid < C ? log_a[row0 + base + tid] : 0.f;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, x, off);
                if (tid >= off) x += y;
            }
            if (base + tid < C) cl[base + tid] = carry + x;
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
    }
    __syncthreads();
    if (tid < C) ce[tid] = expf(cl[C - 1] - cl[tid]);
    // G = K K^T, Gg = Gamma (.) G (strictly lower), QK = Q K^T (lower, diagonal included);
    // Gamma_sr = e^{cl_s - cl_r}
    for (int x = tid; x < C * C; x += NT) {
        const int t = x / C, r = x % C;
        float g = 0.f, a = 0.f;
        if (r <= t) {
            const float* kt = Ks + (size_t)t * ldk;
            const float* kr = Ks + (size_t)r * ldk;
            const float* qt = Qs + (size_t)t * ldk;
            for (int i = 0; i < dk; i++) {
                g += kt[i] * kr[i];
                a += qt[i] * kr[i];
            }
        }
        G[x] = g;
        Gg[x] = r < t ? g * expf(cl[t] - cl[r]) : 0.f;
        QK[x] = a;
    }
    __syncthreads();
    // Lk, Lg by forward substitution, one row per step: threads [0, C) own a column of Lk,
    // threads [C, 2C) a column of Lg
    for (int s = 0; s < C; s++) {
        if (tid < 2 * C) {
            const bool gated = tid >= C;
            const int col = gated ? tid - C : tid;
            float* M = gated ? Lg : Lk;
            const float* A = (gated ? Gg : G) + (size_t)s * C;
            float val;
            if (col > s) {
                val = 0.f;
            } else if (col == s) {
                val = 1.f;
            } else {
                float acc = 0.f;
                for (int r = col; r < s; r++) acc += A[r] * M[(size_t)r * C + col];
                val = -bt[s] * acc;
            }
            M[(size_t)s * C + col] = val;
        }
        __syncthreads();
    }
    // W = Lk diag(beta) K
    for (int x = tid; x < C * dk; x += NT) {
        const int t = x / dk, i = x % dk;
        float acc = 0.f;
        for (int r = 0; r <= t; r++) acc += Lk[(size_t)t * C + r] * bt[r] * Ks[(size_t)r * ldk + i];
        Ws[(size_t)t * ldw + i] = acc;
    }
    __syncthreads();
    const size_t cbase = ((size_t)bh * N + j) * C * dk;
    for (int x = tid; x < C * dk; x += NT) {
        const int t = x / dk, i = x % dk;
        Wg[cbase + x] = Ws[(size_t)t * ldw + i];
        // Q~_t = e^{cl_t} (q_t - sum_{r<=t} (q_t . k_r) w_r)
        float acc = Qs[(size_t)t * ldk + i];
        for (int r = 0; r <= t; r++) acc -= QK[(size_t)t * C + r] * Ws[(size_t)r * ldw + i];
        Qt[cbase + x] = expf(cl[t]) * acc;
    }
    __syncthreads();
    // pseudo-values U = Lg diag(beta) V (over the W buffer); QK <- Gamma (.) QK (diagonal: 1)
    for (int x = tid; x < C * dv; x += NT) {
        const int t = x / dv, jj = x % dv;
        float acc = 0.f;
        for (int r = 0; r <= t; r++) acc += Lg[(size_t)t * C + r] * bt[r] * Vs[(size_t)r * dv + jj];
        Ws[(size_t)t * ldw + jj] = acc;
    }
    for (int x = tid; x < C * C; x += NT) {
        const int t = x / C, r = x % C;
        if (r < t) QK[x] *= expf(cl[t] - cl[r]);
    }
    __syncthreads();
    // attention matrix inside the chunk, lambda-weighted: P[t][s] = lambda_t^(l(t,s)) *
    // beta_s sum_{r=s..t} Gamma_tr (q_t . k_r) Lg[r][s]  (over G, which is no longer needed)
    for (int x = tid; x < C * C; x += NT) {
        const int t = x / C, s = x % C;
        float acc = 0.f;
        if (s <= t) {
            for (int r = s; r <= t; r++) acc += QK[(size_t)t * C + r] * Lg[(size_t)r * C + s];
            const int lvl = fenwick_level(j * C + t, j * C + s);
            acc *= bt[s] * lambda[(row0 + t) * L + lvl];
        }
        G[x] = acc;
    }
    __syncthreads();
    // the chunk's state at its end: K^T diag(e^{cl_end - cl}) U
    if (N > 1) {
        float* node = nodes + ((size_t)bh * node_count + j) * dk * dv;
        for (int x = tid; x < dk * dv; x += NT) {
            const int i = x / dv, jj = x % dv;
            float acc = 0.f;
            for (int s = 0; s < C; s++) acc += Ks[(size_t)s * ldk + i] * ce[s] * Ws[(size_t)s * ldw + jj];
            node[x] = acc;
        }
        if (tid == 0) gam[(size_t)bh * N + j] = expf(cl[C - 1]);
    }
    // in-chunk output P V
    for (int x = tid; x < C * dv; x += NT) {
        const int t = x / dv, jj = x % dv;
        float acc = 0.f;
        for (int s = 0; s <= t; s++) acc += G[(size_t)t * C + s] * Vs[(size_t)s * dv + jj];
        if (N > 1)
            oacc[(row0 + t) * dv + jj] = acc;
        else
            store_f(out + (row0 + t) * dv + jj, acc);
    }
}

// ------------------------------------------------------------------ prefill: one Fenwick level

constexpr int kGdnDS = 16;  // dv columns per level-kernel CTA

// grid (BH * n_even, dv / kGdnDS), 256 threads. CTA (bh, x, slice) takes the x-th read node
// (p, m = 2x) of head bh, columns [16 slice, 16 slice + 16): it reads node m at every chunk
// of block m + 1 and carries it through them; when block m + 1 is complete it writes node
// (p + 1, x) = carried node + node (p, m + 1) if level p + 1 is read.
// Shared memory (fp32): X [dk][16], Y [C][16], and the chunk's Q~, W, K [C][dk + 1] (padded rows).
template <typename T>
__global__ void __launch_bounds__(kGdnThreads) gdn_level_kernel(
    const T* __restrict__ k, const float* __restrict__ Wg, const float* __restrict__ Qt, float* __restrict__ nodes,
    const float* __restrict__ gam, const float* __restrict__ lambda, float* __restrict__ oacc, int T_, int C, int dk,
    int dv, int L, int c_log2, int p, int P, int n_even, int node_count, const __grid_constant__ GdnLevels lo) {
    extern __shared__ float sm[];
    float* X = sm;                        // [dk][16]
    float* Y = X + (size_t)dk * kGdnDS;   // [C][16]
    const int ldk = dk + 1;
    float* Qs = Y + (size_t)C * kGdnDS;   // [C][ldk]
    float* Wsh = Qs + (size_t)C * ldk;    // [C][ldk]
    float* Ksh = Wsh + (size_t)C * ldk;   // [C][ldk]
    const int tid = threadIdx.x;
    const int bh = blockIdx.x / n_even, xi = blockIdx.x % n_even;
    const int j0 = blockIdx.y * kGdnDS;
    const int m = 2 * xi;
    const int N = T_ / C;
    const int span = 1 << p;
    const int b0 = (m + 1) * span;                  // first chunk of the reading block
    const int b1 = min((m + 2) * span, N);          // one past its last chunk
    const bool full = (m + 2) * span <= N;          // block complete: the parent exists
    const bool want_parent = full && p + 1 < P;
    const size_t msz = (size_t)dk * dv;
    const float* src = nodes + ((size_t)bh * node_count + lo.off[p] + m) * msz;
    for (int x = tid; x < dk * kGdnDS; x += kGdnThreads) {
        const int i = x / kGdnDS, d = x % kGdnDS;
        X[x] = src[(size_t)i * dv + j0 + d];
    }
    const int lev = c_log2 + 1 + p;
    for (int jc = b0; jc < b1; jc++) {
        __syncthreads();
        const size_t cbase = ((size_t)bh * N + jc) * C * dk;
        const size_t row0 = (size_t)bh * T_ + (size_t)jc * C;
        for (int x = tid; x < C * dk; x += kGdnThreads) {
            const int pos = (x / dk) * ldk + x % dk;
            Qs[pos] = Qt[cbase + x];
            Wsh[pos] = Wg[cbase + x];
            Ksh[pos] = load_f(k + row0 * dk + x);
        }
        __syncthreads();
        // read: O[t][j0 + d] += lambda_t^(lev) sum_i Q~[t][i] X[i][d]; and Y = W X for the carry
        for (int x = tid; x < C * kGdnDS; x += kGdnThreads) {
            const int t = x / kGdnDS, d = x % kGdnDS;
            float a = 0.f, yw = 0.f;
            for (int i = 0; i < dk; i++) {
                const float xv = X[i * kGdnDS + d];
                a += Qs[(size_t)t * ldk + i] * xv;
                yw += Wsh[(size_t)t * ldk + i] * xv;
            }
            oacc[(row0 + t) * dv + j0 + d] += lambda[(row0 + t) * L + lev] * a;
            Y[x] = yw;
        }
        __syncthreads();
        if (jc + 1 < b1 || want_parent) {
            // carry the node through chunk jc: X <- gamma (X - K^T Y)
            const float gj = gam[(size_t)bh * N + jc];
            for (int x = tid; x < dk * kGdnDS; x += kGdnThreads) {
                const int i = x / kGdnDS, d = x % kGdnDS;
                float acc = 0.f;
                for (int t = 0; t < C; t++) acc += Ksh[(size_t)t * ldk + i] * Y[t * kGdnDS + d];
                X[x] = gj * (X[x] - acc);
            }
        }
    }
    __syncthreads();
    if (want_parent) {
        const float* sib = nodes + ((size_t)bh * node_count + lo.off[p] + m + 1) * msz;
        float* dst = nodes + ((size_t)bh * node_count + lo.off[p + 1] + xi) * msz;
        for (int x = tid; x < dk * kGdnDS; x += kGdnThreads) {
            const int i = x / kGdnDS, d = x % kGdnDS;
            dst[(size_t)i * dv + j0 + d] = X[x] + sib[(size_t)i * dv + j0 + d];
        }
    }
}

template <typename T>
__global__ void gdn_finalize_kernel(const float* __restrict__ oacc, T* __restrict__ out, size_t n) {
    // four elements a thread and step (16-byte loads; 8- or 16-byte stores), then the tail
    const size_t stride = (size_t)gridDim.x * blockDim.x, first = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t n4 = n / 4;
    const float4* src = reinterpret_cast<const float4*>(oacc);
    for (size_t x = first; x < n4; x += stride) {
        const float4 a = src[x];
        if constexpr (sizeof(T) == 2) {
            const __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y), hi = __floats2bfloat162_rn(a.z, a.w);
            uint2 w;
            w.x = *reinterpret_cast<const uint32_t*>(&lo);
            w.y = *reinterpret_cast<const uint32_t*>(&hi);
            reinterpret_cast<uint2*>(out)[x] = w;
        } else {
            reinterpret_cast<float4*>(out)[x] = a;
        }
    }
    for (size_t x = 4 * n4 + first; x < n; x += stride) store_f(out + x, oacc[x]);
}

template <typename T>
cudaError_t gdn_forward_t(const GdnPlan& pl, int dtype, const void* q, const void* k, const void* v,
                          const float* log_a, const float* beta, const float* lambda, void* out, void* workspace,
                          int* err, cudaStream_t stream) {
    const int BH = pl.B * pl.H, C = pl.C, N = pl.N;
    char* ws = static_cast<char*>(workspace);
    float* Wg = reinterpret_cast<float*>(ws + pl.w_off);
    float* Qt = reinterpret_cast<float*>(ws + pl.qt_off);
    float* nodes = reinterpret_cast<float*>(ws + pl.node_off);
    float* gam = reinterpret_cast<float*>(ws + pl.gam_off);
    float* oacc = reinterpret_cast<float*>(ws + pl.oacc_off);
    GdnLevels lo;
    for (int p = 0; p < 32; p++) lo.off[p] = pl.level_off[p];
    const int L = bitlength(static_cast<int64_t>(pl.T) - 1) + 1;
    if (gdn_chunk_tc_supported(pl, dtype)) {
        const cudaError_t e =
            gdn_chunk_tc(pl, q, k, v, log_a, beta, lambda, Wg, Qt, nodes, gam, oacc, out, L, err, stream);
        if (e != cudaSuccess) return e;
    } else {
        const GdnChunkSmem lay(C, pl.dk, pl.dv);
        cudaError_t e = cudaFuncSetAttribute(gdn_chunk_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(lay.total));
        if (e != cudaSuccess) return e;
        gdn_chunk_kernel<T><<<dim3(N, BH), kGdnChunkThreads, lay.total, stream>>>(
            static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), log_a, beta, lambda, Wg, Qt,
            nodes, gam, oacc, static_cast<T*>(out), pl.T, C, pl.dk, pl.dv, L, pl.node_count);
        note_launch(stream, "gdn_chunk");
    }
    if (N == 1) return cudaGetLastError();
    int c_log2 = 0;
    while ((1 << c_log2) < C) c_log2++;
    if (gdn_level_tc_supported(pl, dtype)) {
        const cudaError_t e = gdn_levels_tc(pl, k, Wg, Qt, nodes, gam, lambda, oacc, L, c_log2, err, stream);
        if (e != cudaSuccess) return e;
    } else {
        const size_t smem =
            ((size_t)pl.dk * kGdnDS + (size_t)C * kGdnDS + 3 * (size_t)C * (pl.dk + 1)) * sizeof(float);
        cudaError_t e = cudaFuncSetAttribute(gdn_level_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        for (int p = 0; p < pl.P; p++) {
            const int n_even = (((N - 1) >> p) + 1) / 2;
            if (n_even <= 0) continue;
            gdn_level_kernel<T><<<dim3(BH * n_even, pl.dv / kGdnDS), kGdnThreads, smem, stream>>>(
                static_cast<const T*>(k), Wg, Qt, nodes, gam, lambda, oacc, pl.T, C, pl.dk, pl.dv, L, c_log2, p,
                pl.P, n_even, pl.node_count, lo);
            note_launch(stream, "gdn_level");
        }
    }
    const size_t n = (size_t)BH * pl.T * pl.dv;
    const size_t blocks = (n / 4 + 255) / 256 < 152 * 8 ? (n / 4 + 255) / 256 + 1 : 152 * 8;
    gdn_finalize_kernel<T><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        oacc, static_cast<T*>(out), n);
    note_launch(stream, "gdn_finalize");
    return cudaGetLastError();
}

}  // namespace

bool make_gdn_plan(int B, int H, int T, int dk, int dv, int chunk, GdnPlan* pl) {
    pl->B = B; pl->H = H; pl->T = T; pl->dk = dk; pl->dv = dv;
    pl->C = chunk < 64 ? chunk : 64;
    if (T % pl->C != 0 || dv % kGdnDS != 0) return false;
    pl->N = T / pl->C;
    pl->P = bitlength(static_cast<int64_t>(pl->N) - 1);  // node levels read
    int off = 0;
    for (int p = 0; p < 32; p++) {
        pl->level_off[p] = off;
        if (p <= pl->P) off += pl->N >> p;  // complete nodes of level p
    }
    pl->node_count = off;
    const GdnChunkSmem lay(pl->C, dk, dv);
    if (lay.total > 227 * 1024) return false;
    const size_t BH = (size_t)B * H;
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    pl->w_off = 0;
    pl->qt_off = up(pl->w_off + BH * T * dk * sizeof(float));
    pl->node_off = up(pl->qt_off + BH * T * dk * sizeof(float));
    pl->gam_off = up(pl->node_off + BH * pl->node_count * (size_t)dk * dv * sizeof(float));
    pl->oacc_off = up(pl->gam_off + BH * pl->N * sizeof(float));
    pl->total_bytes = up(pl->oacc_off + BH * T * dv * sizeof(float));
    return true;
}

cudaError_t gdn_forward(const GdnPlan& pl, int dtype, const void* q, const void* k, const void* v,
                        const float* log_a, const float* beta, const float* lambda, void* out, void* workspace,
                        int* err, cudaStream_t stream) {
    return dtype == 0 ? gdn_forward_t<__nv_bfloat16>(pl, dtype, q, k, v, log_a, beta, lambda, out, workspace, err,
                                                     stream)
                      : gdn_forward_t<float>(pl, dtype, q, k, v, log_a, beta, lambda, out, workspace, err, stream);
}

cudaError_t gdn_decode_step(int dtype, const void* q, const void* k, const void* v, const float* log_a,
                            const float* beta, const float* lambda, float* states, const int64_t* t, void* out, int B,
                            int H, int dk, int dv, int Lmax, int* err, cudaStream_t stream) {
    return dtype == 0 ? gdn_decode_t<__nv_bfloat16>(dk, dv, q, k, v, log_a, beta, lambda, states, t, out, B, H, Lmax,
                                                    err, stream)
                      : gdn_decode_t<float>(dk, dv, q, k, v, log_a, beta, lambda, states, t, out, B, H, Lmax, err,
                                            stream);
}

}  // namespace lla
