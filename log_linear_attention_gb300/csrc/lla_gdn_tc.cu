// Tensor-core level pass of the Log-Linear Gated DeltaNet prefill ("Log-Linear Attention",
// pt §2 "Generalização" and §4, fr "Études de Cas": the Fenwick hierarchy of the log-linear
// Mamba-2 applied to the Gated DeltaNet transition A_t = alpha_t (I - beta_t k_t k_t^T)).
//
// Shapes: bf16 k, chunk C = 64, dv = 64, dk in {64, 128} (dk = 64 runs on zero-padded
// operands: the tensor maps of K, W and Q~ have the real dk columns and TMA fills the rest
// with zeros, so every product over dk is the real one and X keeps zero rows dk..127).
//
// One launch per Fenwick level p, one CTA per read node (p, m), m even: the node X (the
// state of chunks [m 2^p, (m+1) 2^p) at their end, dk x dv) is carried through the chunks j
// of the next block. At chunk j, with W_j the WY factor of the chunk's transition product
// (prod over the chunk of (I - beta k k^T) = I - K_j^T W_j, gating a scalar) and Q~_j the
// queries carried back to the chunk start:
//   MMA1 (kind::tf32, M = 128): D = [W_j; Q~_j] X       (rows 0..63: Y = W_j X,
//                                                         rows 64..127: R = Q~_j X)
//   read:  O_t += lambda_t^(level) * Gamma_j * R_t       (fp32 accumulator in HBM)
//   MMA2 (kind::f16, M = 128): X += K_j^T (-Y)           (Y split into bf16 hi + lo)
// X is kept without the chunk decays (X^ <- (I - K^T W) X^); Gamma_j, the product of the
// decays gamma of the chunks already passed, weighs the reads, and the block's node
// (p + 1, m / 2) is Gamma X^ + node (p, m + 1). X lives in TMEM (fp32) and is staged for
// MMA1 as fp32 (read as tf32) in shared memory after every step.
//
// Precision: W_j and Q~_j enter MMA1 as tf32 (10-bit mantissa), X as tf32; Y enters MMA2
// as bf16 hi + lo (16-bit mantissa) against the exact bf16 K; every sum is fp32. A carried
// node accumulates a relative read error near 1e-3 over 64 chunks (against ~1e-2 with bf16
// W, Q~ and X), which keeps the output within the bf16 tolerance.
//
// Every wait is bounded: on overrun the kernel records LLA_ERR_TIMEOUT, lets its own copies
// and MMAs land (bounded), frees its TMEM and returns.
#include "lla_tc_ptx.cuh"

namespace lla {
namespace {

struct GdnTcLevels { int off[32]; };

struct LvCfg {
    static constexpr int kC = 64;                   // chunk tokens
    static constexpr int kDV = 64;
    static constexpr int kAPanel = 16384;           // [W; Q~] fp32: 128 rows x 32 cols
    static constexpr int kA = 0;                    // 4 panels (dk 0..127)
    static constexpr int kKPanel = 8192;            // K bf16: 64 rows x 64 cols
    static constexpr int kK = kA + 4 * kAPanel;     // 2 panels
    static constexpr int kXPanel = 8192;            // X^T fp32: 64 rows (dv) x 32 cols (dk)
    static constexpr int kX = kK + 2 * kKPanel;     // 4 panels; -Y hi, lo (64 x 64 bf16) over the first two
    static constexpr int kBar = kX + 4 * kXPanel;   // mbarriers, TMEM address, failure flag
    static constexpr int kBytes = kBar + 64;
    // the dynamic shared memory base is at least 128-byte aligned; the rest of the 1024-byte
    // alignment the swizzled tiles need comes out of this slack
    static constexpr int kSlack = 1024 - 128;
    static constexpr uint32_t kABytes = 4 * kAPanel;
    static constexpr uint32_t kKBytes = 2 * kKPanel;
};

// Persistent: grid min(chains, 2 per SM), 256 threads (two per TMEM lane, each with half of the
// dv columns), two CTAs per SM.
// A CTA walks the read nodes c = blockIdx.x, blockIdx.x + gridDim.x, ... of level p (chain c:
// head c / n_even, read node m = 2 (c % n_even)), step by step through each chain's chunks. The
// copies of the next step in that walk (the next chunk of the chain, else the first chunk of
// the CTA's next chain) are issued as soon as their buffers are free: [W; Q~] once MMA1 has
// read the stage, K once MMA2 has (or once the step is over, when it needs no MMA2).
__global__ void __launch_bounds__(256, 2)
    gdn_level_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_qt,
                        const __grid_constant__ CUtensorMap tm_k, float* __restrict__ nodes,
                        const float* __restrict__ gam, const float* __restrict__ lambda, float* __restrict__ oacc,
                        int T, int N, int dk, int L, int lev, int p, int P, int node_count, int n_even, int n_chains,
                        const __grid_constant__ GdnTcLevels lo, int* err) {
    using C = LvCfg;
    constexpr int DV = C::kDV;
    constexpr int DH = DV / 2;  // columns of a thread: two threads per TMEM lane
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    uint64_t* full_a = reinterpret_cast<uint64_t*>(smem + C::kBar);
    uint64_t* full_k = full_a + 1;
    uint64_t* mma1 = full_a + 2;
    uint64_t* mma2 = full_a + 3;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full_a + 4);
    volatile int* fail = reinterpret_cast<volatile int*>(full_a + 5);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row = tid & 127;   // TMEM lane: a dk row of X, a token row of Y (< 64) or of R
    const int half = tid >> 7;   // which DH columns of the row
    const int wq = warp & 3;     // lane quadrant of this warp
    if (pad > static_cast<uint32_t>(C::kSlack)) {  // base alignment below the assumed 128 bytes
        if (tid == 0) record_error(err, kDevBadInput);
        return;
    }
    const int span = 1 << p;
    const size_t msz = static_cast<size_t>(dk) * DV;
    auto chain_range = [&](int c, int& bh, int& xi, int& b0, int& b1) {
        bh = c / n_even;
        xi = c - bh * n_even;
        b0 = (2 * xi + 1) * span;
        b1 = min((2 * xi + 2) * span, N);
    };
    auto node_ptr = [&](int bh, int lvl, int idx) {
        return nodes + (static_cast<size_t>(bh) * node_count + lo.off[lvl] + idx) * msz;
    };

    if (tid == 0) {
        mbar_init(full_a, 1);
        mbar_init(full_k, 1);
        mbar_init(mma1, 1);
        mbar_init(mma2, 1);
        fence_mbar_init();
        *fail = 0;
    }
    if (warp == 0) tmem_alloc(tmem_slot, 128);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tD = tmem + lane_base;       // MMA1 result, columns [0, 64)
    const uint32_t tX = tmem + lane_base + 64;  // carried node, columns [64, 128)
    constexpr uint32_t kIdA = idesc_tf32(128, DV);        // [W; Q~] (K-major) x X (K-major)
    constexpr uint32_t kIdB = idesc_bf16(128, DV, 1, 1);  // K^T (MN-major) x Y (MN-major)

    int n_a = 0, n_k = 0, n_m1 = 0, n_m2 = 0;  // copies and MMA groups issued (thread 0)
    auto load_a = [&](int c, int jc) {
        const int r = ((c / n_even) * N + jc) * C::kC;
        mbar_expect_tx(full_a, C::kABytes);
#pragma unroll
        for (int q = 0; q < 4; q++) {
            tma_load_2d(smem + C::kA + q * C::kAPanel, &tm_w, full_a, 32 * q, r);
            tma_load_2d(smem + C::kA + q * C::kAPanel + C::kAPanel / 2, &tm_qt, full_a, 32 * q, r);
        }
        n_a++;
    };
    auto load_k = [&](int c, int jc) {
        const int r = (c / n_even) * T + jc * C::kC;
        mbar_expect_tx(full_k, C::kKBytes);
        tma_load_2d(smem + C::kK, &tm_k, full_k, 0, r);
        tma_load_2d(smem + C::kK + C::kKPanel, &tm_k, full_k, 64, r);
        n_k++;
    };
    // the step after (chain c, chunk jc) in this CTA's walk; false at the end of the walk
    auto next_step = [&](int c, int jc, int& nc, int& njc) -> bool {
        int bh, xi, b0, b1;
        chain_range(c, bh, xi, b0, b1);
        if (jc + 1 < b1) {
            nc = c;
            njc = jc + 1;
            return true;
        }
        nc = c + gridDim.x;
        if (nc >= n_chains) return false;
        chain_range(nc, bh, xi, b0, b1);
        njc = b0;
        return true;
    };
    // thread 0 waits; the block learns the outcome from `fail` after its next barrier
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (mbar_wait(bar, parity)) return true;
        *fail = 1;
        record_error(err, kDevTimeout);
        return false;
    };
    // X row i (i = row, a dk row; this thread's DH columns d) into the K-major fp32 staging of
    // X^T: element (d, i) sits in panel i / 32, row d, 16-byte chunk ((i % 32) / 4) ^ (d % 8),
    // word i % 4
    auto stage_xt = [&](const float* x) {
        uint8_t* base = smem + C::kX + (row >> 5) * C::kXPanel + (row & 3) * 4;
        const int c = (row & 31) >> 2;
#pragma unroll
        for (int e = 0; e < DH; e++) {
            const int d = DH * half + e;
            *reinterpret_cast<float*>(base + d * 128 + ((c ^ (d & 7)) << 4)) = x[e];
        }
    };

    // This thread's DH columns of row-major fp32 rows of DV values, one row per thread of a warp
    // with consecutive rows (`rows` points at the warp's first row, `live` rows exist): loaded
    // and stored in whole 64-byte runs of 8 rows per warp access, the chunks swapped within lane
    // groups.
    auto load_rows = [&](const float* rows, int live, float* x) {
        const int g0 = lane & ~3, c = lane & 3;
#pragma unroll
        for (int q = 0; q < DH / 16; q++) {
            uint4 y[4];
#pragma unroll
            for (int i = 0; i < 4; i++)
                y[i] = g0 + i < live
                           ? *reinterpret_cast<const uint4*>(rows + (g0 + i) * DV + DH * half + 16 * q + 4 * c)
                           : make_uint4(0u, 0u, 0u, 0u);
            lane_group_transpose(y, lane);
#pragma unroll
            for (int j = 0; j < 4; j++) {
                x[16 * q + 4 * j] = __uint_as_float(y[j].x);
                x[16 * q + 4 * j + 1] = __uint_as_float(y[j].y);
                x[16 * q + 4 * j + 2] = __uint_as_float(y[j].z);
                x[16 * q + 4 * j + 3] = __uint_as_float(y[j].w);
            }
        }
    };
    auto store_rows = [&](float* rows, int live, const float* x) {
        const int g0 = lane & ~3, c = lane & 3;
#pragma unroll
        for (int q = 0; q < DH / 16; q++) {
            uint4 y[4];
#pragma unroll
            for (int j = 0; j < 4; j++)
                y[j] = make_uint4(__float_as_uint(x[16 * q + 4 * j]), __float_as_uint(x[16 * q + 4 * j + 1]),
                                  __float_as_uint(x[16 * q + 4 * j + 2]), __float_as_uint(x[16 * q + 4 * j + 3]));
            lane_group_transpose(y, lane);
#pragma unroll
            for (int i = 0; i < 4; i++)
                if (g0 + i < live) *reinterpret_cast<uint4*>(rows + (g0 + i) * DV + DH * half + 16 * q + 4 * c) = y[i];
        }
    };

    if (tid == 0 && static_cast<int>(blockIdx.x) < n_chains) {
        int bh, xi, b0, b1;
        chain_range(blockIdx.x, bh, xi, b0, b1);
        load_a(blockIdx.x, b0);
        load_k(blockIdx.x, b0);
    }
    int gs = 0;  // steps taken: the phase of full_a, full_k and mma1
    for (int c = blockIdx.x; c < n_chains; c += gridDim.x) {
        int bh, xi, b0, b1;
        chain_range(c, bh, xi, b0, b1);
        const int m = 2 * xi;
        const bool want_parent = (m + 2) * span <= N && p + 1 < P;
        if (tid == 0 && c + static_cast<int>(gridDim.x) < n_chains) {
            // the next chain's node and sibling into L2 while this chain runs
            int nbh, nxi, nb0, nb1;
            chain_range(c + gridDim.x, nbh, nxi, nb0, nb1);
            prefetch_l2(node_ptr(nbh, p, 2 * nxi), static_cast<uint32_t>(msz * 4));
            if ((2 * nxi + 2) * span <= N && p + 1 < P)
                prefetch_l2(node_ptr(nbh, p, 2 * nxi + 1), static_cast<uint32_t>(msz * 4));
        }
        {
            // X = node (p, m); rows dk..127 are zero
            float x[DH];
            load_rows(node_ptr(bh, p, m) + static_cast<size_t>(32 * wq) * DV, dk - 32 * wq, x);
            tmem_st32(tX + DH * half, x);
            stage_xt(x);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        float Gam = 1.f;  // product of gamma over the chunks passed
        for (int jc = b0; jc < b1; jc++, gs++) {
            const uint32_t ph = gs & 1;
            const bool last = jc + 1 == b1;
            const bool carry = !last || want_parent;
            int nc = 0, njc = 0;
            const bool more = next_step(c, jc, nc, njc);
            const size_t row0 = static_cast<size_t>(bh) * T + static_cast<size_t>(jc) * C::kC;
            // the read's lambda and accumulator row, loaded while MMA1 runs
            float lw = 0.f;
            float oa[DH];
            if (row >= C::kC) {  // warps 2, 3, 6 and 7 whole
                const size_t t = row0 + (row - C::kC);
                lw = lambda[t * L + lev] * Gam;
                load_rows(oacc + (row0 + 32 * (wq - 2)) * DV, 32, oa);
            }
            if (tid == 0 && wait(full_a, ph)) {
                tc_fence_after();
                const uint32_t ab = smem_u32(smem + C::kA), xb = smem_u32(smem + C::kX);
#pragma unroll
                for (int kk = 0; kk < 16; kk++) {
                    const uint32_t oa_ = (kk >> 2) * C::kAPanel + (kk & 3) * 32;
                    const uint32_t ob = (kk >> 2) * C::kXPanel + (kk & 3) * 32;
                    mma_tf32(tmem, sdesc(ab + oa_, 16, 1024), sdesc(xb + ob, 16, 1024), kIdA, kk > 0 ? 1u : 0u);
                }
                mma_commit(mma1);
                n_m1++;
                if (wait(mma1, ph) && more) load_a(nc, njc);  // MMA1 has read the stage
            }
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            if (*fail) break;
            float v[DH];
            tmem_ld32(tD + DH * half, v);
            if (row < C::kC) {
                if (carry) {
                    // -Y row `row` as bf16 hi + lo, MN-major rows of 64 dv (one 128-byte row per
                    // token; this thread's DH columns are chunks 4 half .. 4 half + 3)
                    uint8_t* hi = smem + C::kX;
                    uint8_t* lo_ = smem + C::kX + C::kXPanel;
#pragma unroll
                    for (int c8 = 0; c8 < DH / 8; c8++) {
                        uint32_t h[4], l[4];
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            const float a = -v[8 * c8 + 2 * e], b = -v[8 * c8 + 2 * e + 1];
                            h[e] = pack_bf16(a, b);
                            const float2 hf = unpack_bf16(h[e]);
                            l[e] = pack_bf16(a - hf.x, b - hf.y);
                        }
                        const int ch = (DH / 8) * half + c8;
                        *reinterpret_cast<uint4*>(hi + sw128_off(row, ch)) = make_uint4(h[0], h[1], h[2], h[3]);
                        *reinterpret_cast<uint4*>(lo_ + sw128_off(row, ch)) = make_uint4(l[0], l[1], l[2], l[3]);
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < DH; e++) oa[e] = fmaf(lw, v[e], oa[e]);
                store_rows(oacc + (row0 + 32 * (wq - 2)) * DV, 32, oa);
            }
            if (!carry) {
                // no MMA2: K of this step arrived unused; the next step's K may take its buffer
                if (tid == 0 && wait(full_k, ph) && more) load_k(nc, njc);
                tc_fence_before();
                __syncthreads();
                tc_fence_after();
                gs++;
                break;
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            if (tid == 0 && wait(full_k, ph)) {
                tc_fence_after();
                const uint32_t kb = smem_u32(smem + C::kK), yb = smem_u32(smem + C::kX);
#pragma unroll
                for (int kk = 0; kk < C::kC / 16; kk++)
#pragma unroll
                    for (int h = 0; h < 2; h++)
                        mma_bf16(tmem + 64, sdesc(kb + kk * 2048, C::kKPanel, 1024),
                                 sdesc(yb + h * C::kXPanel + kk * 2048, C::kXPanel, 1024), kIdB, 1u);
                mma_commit(mma2);
                n_m2++;
                if (wait(mma2, (n_m2 - 1) & 1) && more) load_k(nc, njc);  // MMA2 has read K
            }
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            if (*fail) break;
            Gam *= gam[static_cast<size_t>(bh) * N + jc];
            tmem_ld32(tX + DH * half, v);
            if (!last) {
                stage_xt(v);
            } else {
                // node (p + 1, m / 2) = Gamma X^ + node (p, m + 1) (rows dk.. do not exist)
                float sib[DH];
                load_rows(node_ptr(bh, p, m + 1) + static_cast<size_t>(32 * wq) * DV, dk - 32 * wq, sib);
#pragma unroll
                for (int e = 0; e < DH; e++) sib[e] = fmaf(Gam, v[e], sib[e]);
                store_rows(node_ptr(bh, p + 1, xi) + static_cast<size_t>(32 * wq) * DV, dk - 32 * wq, sib);
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
        }
        if (*fail) break;
    }

    if (tid == 0 && *fail) {
        // let this CTA's copies and MMAs land before its shared memory and TMEM are released
        if (n_a > 0) mbar_wait(full_a, (n_a - 1) & 1);
        if (n_k > 0) mbar_wait(full_k, (n_k - 1) & 1);
        if (n_m1 > 0) mbar_wait(mma1, (n_m1 - 1) & 1);
        if (n_m2 > 0) mbar_wait(mma2, (n_m2 - 1) & 1);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// ------------------------------------------------------------------ chunk pass

struct CkCfg {
    static constexpr int kC = 64;                   // chunk tokens
    static constexpr int kDV = 64;
    static constexpr int kKQPanel = 16384;          // 128 rows x 64 dk (bf16): rows 0..63 K, 64..127 Q
    static constexpr int kKQ = 0;                   // 2 panels (dk 0..127)
    static constexpr int kV = kKQ + 2 * kKQPanel;   // V: 64 rows x 64 dv (bf16), 8 KB
    static constexpr int kA2 = kV + 8192;           // A2 hi, lo: 128 rows x 64 tokens (bf16), 16 KB each
    static constexpr int kR = kA2 + 32768;          // Bk, Bg (fp32 [64][kLd]); later A1 hi, lo; later U hi, lo
    static constexpr int kLd = 68;                  // row stride of Bk, Bg in floats (16-byte rows, no bank conflicts)
    static constexpr int kBBytes = 64 * kLd * 4;
    static constexpr int kRBytes = 2 * kBBytes > 32768 ? 2 * kBBytes : 32768;
    static constexpr int kScal = kR + kRBytes;      // cl, beta, ce: 64 floats each
    static constexpr int kBar = kScal + 3 * 64 * 4;
    static constexpr int kBytes = kBar + 64;
    static constexpr int kSlack = 1024 - 128;
    static constexpr uint32_t kInBytes = 2 * kKQPanel + 8192;
};

// grid (N chunks, B*H), 256 threads (warp w reads TMEM lanes 32 (w % 4) ..), two CTAs per SM.
// Per chunk of 64 tokens:
//   MMA-a: [K; Q] K^T -> G = K K^T, QK = Q K^T (bf16 operands, exact products)
//   Bk = diag(beta) strictlower(G), Bg = diag(beta) strictlower(Gamma (.) G), Gamma_tr = e^{cl_t - cl_r}
//   Lk = (I + Bk)^-1, Lg = (I + Bg)^-1 in fp32, blockwise in place (16 x 16 diagonal blocks by row
//   solves, then two merges in rolled loops: the kernel's code stays compact, which keeps its
//   warps fed by the instruction cache)
//   MMA-m: [tril(QK); Z] [Lk | Lg] -> tril(QK) Lk and Z Lg, Z = tril(Gamma (.) QK)
//   MMA-b: [Lk diag(beta); tril(QK) Lk diag(beta)] K -> W = Lk diag(beta) K and the correction of
//          Q~ = diag(e^{cl}) (Q - tril(QK) W)
//   MMA-c: [Lg diag(beta); P] V -> U = Lg diag(beta) V and the in-chunk output P V, with
//          P[t][s] = lambda_t^(level(t,s)) (Z Lg)[t][s] beta_s for s <= t
//   MMA-d: K^T diag(e^{cl_end - cl}) U -> the chunk's state, node (0, j)
// Every fp32 operand of MMA-m/b/c/d is split into bf16 hi + lo (MMA-m: three passes, the others
// two); K and V are exact in bf16.
__global__ void __launch_bounds__(256, 2)
    gdn_chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_w,
                        const __grid_constant__ CUtensorMap tm_qt, const __nv_bfloat16* __restrict__ q,
                        const float* __restrict__ log_a, const float* __restrict__ beta,
                        const float* __restrict__ lambda, float* __restrict__ Wg, float* __restrict__ Qt,
                        float* __restrict__ nodes, float* __restrict__ gam, float* __restrict__ oacc,
                        __nv_bfloat16* __restrict__ out, int T, int N, int dk, int L, int node_count, int* err) {
    using C = CkCfg;
    constexpr int DV = C::kDV;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    float* Bk = reinterpret_cast<float*>(smem + C::kR);
    float* Bg = Bk + 64 * C::kLd;
    float* cl = reinterpret_cast<float*>(smem + C::kScal);
    float* bt = cl + 64;
    float* ce = bt + 64;
    uint64_t* in_full = reinterpret_cast<uint64_t*>(smem + C::kBar);
    uint64_t* mma_a = in_full + 1;
    uint64_t* mma_bc = in_full + 2;
    uint64_t* mma_d = in_full + 3;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(in_full + 4);
    volatile int* fail = reinterpret_cast<volatile int*>(in_full + 5);
    uint64_t* mma_m = in_full + 6;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (pad > static_cast<uint32_t>(C::kSlack)) {
        if (tid == 0) record_error(err, kDevBadInput);
        return;
    }
    const int j = blockIdx.x, bh = blockIdx.y;
    const size_t row0 = static_cast<size_t>(bh) * T + static_cast<size_t>(j) * C::kC;
    const int t = tid & 63;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;

    if (tid == 0) {
        mbar_init(in_full, 1);
        mbar_init(mma_a, 1);
        mbar_init(mma_bc, 1);
        mbar_init(mma_d, 1);
        mbar_init(mma_m, 1);
        fence_mbar_init();
        *fail = 0;
    }
    if (warp == 0) tmem_alloc(tmem_slot, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    int n_in = 0, n_a = 0, n_bc = 0, n_d = 0, n_m = 0, n_st = 0;
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (mbar_wait(bar, parity)) return true;
        *fail = 1;
        record_error(err, kDevTimeout);
        return false;
    };
    auto block_sync = [&]() {
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };

    if (tid == 0) {
        mbar_expect_tx(in_full, C::kInBytes);
        for (int pnl = 0; pnl < 2; pnl++) {
            tma_load_2d(smem + C::kKQ + pnl * C::kKQPanel, &tm_k, in_full, 64 * pnl, static_cast<int>(row0));
            tma_load_2d(smem + C::kKQ + pnl * C::kKQPanel + C::kKQPanel / 2, &tm_q, in_full, 64 * pnl,
                        static_cast<int>(row0));
        }
        tma_load_2d(smem + C::kV, &tm_v, in_full, 0, static_cast<int>(row0));
        n_in = 1;
    }
    if (warp == 1) {
        // in-chunk inclusive prefix of log a (natural log units)
        float a0 = log_a[row0 + lane], a1 = log_a[row0 + 32 + lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y0 = __shfl_up_sync(0xffffffffu, a0, off), y1 = __shfl_up_sync(0xffffffffu, a1, off);
            if (lane >= off) {
                a0 += y0;
                a1 += y1;
            }
        }
        const float tot0 = __shfl_sync(0xffffffffu, a0, 31);
        cl[lane] = a0;
        cl[32 + lane] = a1 + tot0;
    }
    if (warp == 2) {
        bt[lane] = beta[row0 + lane];
        bt[32 + lane] = beta[row0 + 32 + lane];
    }
    __syncthreads();
    if (tid < 64) ce[tid] = expf(cl[63] - cl[tid]);
    do {
        if (tid == 0 && wait(in_full, 0)) {
            tc_fence_after();
            const uint32_t kq = smem_u32(smem + C::kKQ);
#pragma unroll
            for (int kk = 0; kk < 8; kk++) {
                const uint32_t off = (kk >> 2) * C::kKQPanel + (kk & 3) * 32;
                mma_bf16(tmem, sdesc(kq + off, 16, 1024), sdesc(kq + off, 16, 1024), idesc_bf16(128, 64, 0, 0),
                         kk > 0 ? 1u : 0u);
            }
            mma_commit(mma_a);
            n_a = 1;
            wait(mma_a, 0);
        }
        block_sync();
        if (*fail) break;

        // ---- G, QK out of TMEM (decay factors 2^((cl_t - cl_r) log2 e) have non-positive
        //      exponents, r <= t).
        //      Lanes 0..63 (warps 0, 1: columns 0..31; warps 4, 5: 32..63): Bk = diag(beta)
        //      strictlower(G) and Bg = diag(beta) strictlower(Gamma (.) G), fp32 in the R area.
        //      Lanes 64..127: the A operand of MMA-m, [tril(QK); Z] with Z = tril(Gamma (.) QK),
        //      as bf16 hi + lo K-major rows of 64 tokens in the A2 area (warps 2, 3: tril(QK)
        //      rows; warps 6, 7: Z rows).
        const float clt = cl[t] * kLog2e;
        if ((warp & 3) < 2) {
            const int h = warp >> 2;  // column half
            float x[32];
            tmem_ld32(tmem + lane_base + 32 * h, x);
            const float b = bt[t];
            float4* bk = reinterpret_cast<float4*>(Bk + t * C::kLd + 32 * h);
            float4* bg = reinterpret_cast<float4*>(Bg + t * C::kLd + 32 * h);
#pragma unroll
            for (int r4 = 0; r4 < 8; r4++) {
                float vk[4], vg[4];
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const int r = 32 * h + 4 * r4 + e;
                    const float g = x[4 * r4 + e];
                    vk[e] = r < t ? b * g : 0.f;
                    vg[e] = r < t ? b * ex2_ftz(clt - cl[r] * kLog2e) * g : 0.f;
                }
                bk[r4] = make_float4(vk[0], vk[1], vk[2], vk[3]);
                bg[r4] = make_float4(vg[0], vg[1], vg[2], vg[3]);
            }
        } else {
            const bool zrow = warp >= 4;
            const int row = zrow ? 64 + t : t;
            uint8_t* dst = smem + C::kA2;
#pragma unroll 1
            for (int hh = 0; hh < 2; hh++) {
                float x[32];
                tmem_ld32(tmem + lane_base + 32 * hh, x);
#pragma unroll
                for (int c8 = 0; c8 < 4; c8++) {
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        float w2[2];
#pragma unroll
                        for (int u = 0; u < 2; u++) {
                            const int r = 32 * hh + 8 * c8 + 2 * e + u;
                            const float q = x[8 * c8 + 2 * e + u];
                            const float w = zrow ? q * ex2_ftz(clt - cl[r] * kLog2e) : q;
                            w2[u] = r <= t ? w : 0.f;
                        }
                        hi[e] = pack_bf16(w2[0], w2[1]);
                        const float2 hf = unpack_bf16(hi[e]);
                        lo[e] = pack_bf16(w2[0] - hf.x, w2[1] - hf.y);
                    }
                    const int c = 4 * hh + c8;
                    *reinterpret_cast<uint4*>(dst + sw128_off(row, c)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4*>(dst + 16384 + sw128_off(row, c)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
            }
        }
        __syncthreads();

        // ---- Lk = (I + Bk)^-1 (threads 0..127) and Lg = (I + Bg)^-1 (threads 128..255), in place,
        //      by blocks: the 16 x 16 diagonal blocks by row solves, then pairs of blocks merged,
        //      [[A, 0], [C, D]]^-1 = [[A^-1, 0], [-D^-1 C A^-1, D^-1]], into 32 x 32 and 64 x 64.
        //      The merge products run in rolled loops; their C A^-1 goes to a scratch in the Q
        //      half of the input tile (Q is not read after MMA-a). B is strictly lower, so every
        //      block above the diagonal is zero throughout.
        {
            const int mt = tid & 127;
            float* Bm = tid < 128 ? Bk : Bg;
            float* tsc = reinterpret_cast<float*>(smem + C::kKQ + (tid < 128 ? 0 : C::kKQPanel) + C::kKQPanel / 2);
            if (mt < 64) {
                // row i of the inverse of diagonal block b (its right-hand side e_i is zero past i)
                const int b16 = (mt >> 4) * 16, i = mt & 15;
                float y[16];
#pragma unroll
                for (int c = 0; c < 16; c++) y[c] = c == i ? 1.f : 0.f;
#pragma unroll
                for (int s = 15; s > 0; s--) {
                    if (s > i) continue;
                    const float ys = y[s];
                    const float* brow = Bm + (b16 + s) * C::kLd + b16;
#pragma unroll
                    for (int c = 0; c < s; c++) y[c] = fmaf(-ys, brow[c], y[c]);
                }
                __syncwarp();  // the block's rows are read by the warp that holds them
                float4* out = reinterpret_cast<float4*>(Bm + (b16 + i) * C::kLd + b16);
#pragma unroll
                for (int c4 = 0; c4 < 4; c4++) out[c4] = make_float4(y[4 * c4], y[4 * c4 + 1], y[4 * c4 + 2], y[4 * c4 + 3]);
            }
            __syncthreads();
            // 16 -> 32: blocks (2c, 2c + 1), rows r0 = 32 c ..; thread: row i, columns j0 .. j0 + 3
            {
                const int c = mt >> 6, i = (mt >> 2) & 15, j0 = (mt & 3) * 4, r0 = 32 * c;
                float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 4
                for (int k = 0; k < 16; k++) {
                    const float bik = Bm[(r0 + 16 + i) * C::kLd + r0 + k];
                    const float4 d = *reinterpret_cast<const float4*>(Bm + (r0 + k) * C::kLd + r0 + j0);
                    a0 = fmaf(bik, d.x, a0); a1 = fmaf(bik, d.y, a1); a2 = fmaf(bik, d.z, a2); a3 = fmaf(bik, d.w, a3);
                }
                *reinterpret_cast<float4*>(tsc + (c * 16 + i) * 16 + j0) = make_float4(a0, a1, a2, a3);
            }
            __syncthreads();
            {
                const int c = mt >> 6, i = (mt >> 2) & 15, j0 = (mt & 3) * 4, r0 = 32 * c;
                float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 4
                for (int k = 0; k <= i; k++) {
                    const float dik = Bm[(r0 + 16 + i) * C::kLd + r0 + 16 + k];
                    const float4 v = *reinterpret_cast<const float4*>(tsc + (c * 16 + k) * 16 + j0);
                    a0 = fmaf(-dik, v.x, a0); a1 = fmaf(-dik, v.y, a1); a2 = fmaf(-dik, v.z, a2); a3 = fmaf(-dik, v.w, a3);
                }
                *reinterpret_cast<float4*>(Bm + (r0 + 16 + i) * C::kLd + r0 + j0) = make_float4(a0, a1, a2, a3);
            }
            __syncthreads();
            // 32 -> 64: thread: row i of the lower half, columns j0 .. j0 + 7
            {
                const int i = mt >> 2, j0 = (mt & 3) * 8;
                float a[8];
#pragma unroll
                for (int e = 0; e < 8; e++) a[e] = 0.f;
#pragma unroll 4
                for (int k = 0; k < 32; k++) {
                    const float bik = Bm[(32 + i) * C::kLd + k];
                    const float4 d0 = *reinterpret_cast<const float4*>(Bm + k * C::kLd + j0);
                    const float4 d1 = *reinterpret_cast<const float4*>(Bm + k * C::kLd + j0 + 4);
                    a[0] = fmaf(bik, d0.x, a[0]); a[1] = fmaf(bik, d0.y, a[1]); a[2] = fmaf(bik, d0.z, a[2]);
                    a[3] = fmaf(bik, d0.w, a[3]); a[4] = fmaf(bik, d1.x, a[4]); a[5] = fmaf(bik, d1.y, a[5]);
                    a[6] = fmaf(bik, d1.z, a[6]); a[7] = fmaf(bik, d1.w, a[7]);
                }
                *reinterpret_cast<float4*>(tsc + i * 32 + j0) = make_float4(a[0], a[1], a[2], a[3]);
                *reinterpret_cast<float4*>(tsc + i * 32 + j0 + 4) = make_float4(a[4], a[5], a[6], a[7]);
            }
            __syncthreads();
            {
                const int i = mt >> 2, j0 = (mt & 3) * 8;
                float a[8];
#pragma unroll
                for (int e = 0; e < 8; e++) a[e] = 0.f;
#pragma unroll 4
                for (int k = 0; k <= i; k++) {
                    const float dik = Bm[(32 + i) * C::kLd + 32 + k];
                    const float4 v0 = *reinterpret_cast<const float4*>(tsc + k * 32 + j0);
                    const float4 v1 = *reinterpret_cast<const float4*>(tsc + k * 32 + j0 + 4);
                    a[0] = fmaf(-dik, v0.x, a[0]); a[1] = fmaf(-dik, v0.y, a[1]); a[2] = fmaf(-dik, v0.z, a[2]);
                    a[3] = fmaf(-dik, v0.w, a[3]); a[4] = fmaf(-dik, v1.x, a[4]); a[5] = fmaf(-dik, v1.y, a[5]);
                    a[6] = fmaf(-dik, v1.z, a[6]); a[7] = fmaf(-dik, v1.w, a[7]);
                }
                float4* out = reinterpret_cast<float4*>(Bm + (32 + i) * C::kLd + j0);
                out[0] = make_float4(a[0], a[1], a[2], a[3]);
                out[1] = make_float4(a[4], a[5], a[6], a[7]);
            }
            __syncthreads();
        }

        // ---- MMA-m: [tril(QK); Z] [Lk | Lg] -> tril(QK) Lk (rows 0..63, columns 0..63) and Z Lg
        //      (rows 64..127, columns 64..127), 3 bf16 passes (hi hi, hi lo, lo hi). Thread
        //      (m = tid / 128, row r, half hl) keeps L_m[r][32 hl ..] for the A operands; B =
        //      [Lk | Lg] (MN-major, 64-column atoms: Lk, Lg) is written over the R area.
        const int lm = tid >> 7, lr = (tid >> 1) & 63, hl = tid & 1;
        float lv[32];
        {
            const float4* src = reinterpret_cast<const float4*>((lm ? Bg : Bk) + lr * C::kLd + 32 * hl);
#pragma unroll
            for (int c4 = 0; c4 < 8; c4++) {
                const float4 f = src[c4];
                lv[4 * c4] = f.x; lv[4 * c4 + 1] = f.y; lv[4 * c4 + 2] = f.z; lv[4 * c4 + 3] = f.w;
            }
        }
        __syncthreads();
        {
            uint8_t* dst = smem + C::kR + lm * 8192;
#pragma unroll
            for (int c8 = 0; c8 < 4; c8++) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const float a = lv[8 * c8 + 2 * e], b2 = lv[8 * c8 + 2 * e + 1];
                    hi[e] = pack_bf16(a, b2);
                    const float2 hf = unpack_bf16(hi[e]);
                    lo[e] = pack_bf16(a - hf.x, b2 - hf.y);
                }
                *reinterpret_cast<uint4*>(dst + sw128_off(lr, 4 * hl + c8)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(dst + 16384 + sw128_off(lr, 4 * hl + c8)) =
                    make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
        fence_async_smem();
        block_sync();
        if (tid == 0) {
            const uint32_t ab = smem_u32(smem + C::kA2), bb = smem_u32(smem + C::kR);
#pragma unroll
            for (int pass = 0; pass < 3; pass++) {
                const uint32_t pa = pass == 2 ? 16384u : 0u, pb = pass == 1 ? 16384u : 0u;
#pragma unroll
                for (int kk = 0; kk < 4; kk++)
                    mma_bf16(tmem + 64, sdesc(ab + pa + kk * 32, 16, 1024), sdesc(bb + pb + kk * 2048, 8192, 1024),
                             idesc_bf16(128, 128, 0, 1), (pass > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(mma_m);
            n_m = 1;
            wait(mma_m, 0);
        }
        block_sync();
        if (*fail) break;

        // ---- A operands, bf16 hi + lo, K-major rows of 64 tokens: A1 = [Lk; tril(QK) Lk] diag(beta)
        //      over the R area, A2 = [Lg diag(beta); P] over the A2 area, with
        //      P[t][s] = lambda_t^(level(t,s)) (Z Lg)[t][s] beta_s for s <= t.
        {
            // product row t (lane), columns 32 hq ..: tril(QK) Lk (lanes 0..63) or Z Lg (lanes 64..127)
            const int hq = warp >> 2;
            const bool zq = (warp & 3) >= 2;
            float pv[32];
            tmem_ld32(tmem + lane_base + 64 + (zq ? 64 : 0) + 32 * hq, pv);
            float lam[7];
            if (zq) {
#pragma unroll
                for (int l = 0; l < 7; l++) lam[l] = lambda[(row0 + t) * L + l];
            }
            // (tmask >= 0: the row is token tmask's row of P: lambda weights and the causal mask)
            auto put = [&](uint8_t* dst, int row, int c0, const float* v, int tmask) {
#pragma unroll
                for (int c8 = 0; c8 < 4; c8++) {
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        float w2[2];
#pragma unroll
                        for (int u = 0; u < 2; u++) {
                            const int s = c0 + 8 * c8 + 2 * e + u;
                            float w = v[8 * c8 + 2 * e + u] * bt[s];
                            if (tmask >= 0) {
                                const int xo = tmask ^ s;
                                float lw = xo >= 32 ? lam[6] : lam[5];
                                lw = xo < 16 ? lam[4] : lw;
                                lw = xo < 8 ? lam[3] : lw;
                                lw = xo < 4 ? lam[2] : lw;
                                lw = xo < 2 ? lam[1] : lw;
                                lw = xo == 0 ? lam[0] : lw;
                                w = s <= tmask ? w * lw : 0.f;
                            }
                            w2[u] = w;
                        }
                        hi[e] = pack_bf16(w2[0], w2[1]);
                        const float2 hf = unpack_bf16(hi[e]);
                        lo[e] = pack_bf16(w2[0] - hf.x, w2[1] - hf.y);
                    }
                    const int cc = (c0 >> 3) + c8;
                    *reinterpret_cast<uint4*>(dst + sw128_off(row, cc)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4*>(dst + 16384 + sw128_off(row, cc)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
            };
            // (MMA-m has completed: its operands in the R and A2 areas are free)
            put(smem + (lm ? C::kA2 : C::kR), lr, 32 * hl, lv, -1);
            put(smem + (zq ? C::kA2 : C::kR), 64 + t, 32 * hq, pv, zq ? t : -1);
        }
        fence_async_smem();
        block_sync();
        if (tid == 0) {
            const uint32_t kq = smem_u32(smem + C::kKQ), a1 = smem_u32(smem + C::kR), a2 = smem_u32(smem + C::kA2),
                           vb = smem_u32(smem + C::kV);
#pragma unroll
            for (int kk = 0; kk < 4; kk++)
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const uint32_t acc = (kk > 0 || h > 0) ? 1u : 0u;
                    mma_bf16(tmem + 64, sdesc(a1 + h * 16384 + kk * 32, 16, 1024),
                             sdesc(kq + kk * 2048, C::kKQPanel, 1024), idesc_bf16(128, 128, 0, 1), acc);
                    mma_bf16(tmem + 192, sdesc(a2 + h * 16384 + kk * 32, 16, 1024), sdesc(vb + kk * 2048, 8192, 1024),
                             idesc_bf16(128, 64, 0, 1), acc);
                }
            mma_commit(mma_bc);
            n_bc = 1;
            wait(mma_bc, 0);
        }
        block_sync();
        if (*fail) break;

        // ---- W, Q~ (fp32, the level pass reads them), U (into shared memory), in-chunk output
        auto qt_box = [&](int b) -> uint8_t* {
            return b < 2 ? smem + C::kKQ + b * C::kKQPanel + C::kKQPanel / 2 : smem + C::kR + 16384 + (b - 2) * 8192;
        };
        {
            const int half = warp >> 2;  // which 64 of the 128 columns of MMA-b, 32 of the 64 of MMA-c
            const bool top = (warp & 3) < 2;  // TMEM lanes 0..63 (W, U rows) or 64..127 (Q~, output rows)
            float v[64];
            tmem_ld32(tmem + lane_base + 64 + 64 * half, v);
            tmem_ld32(tmem + lane_base + 96 + 64 * half, v + 32);
            if (N > 1 && 64 * half < dk) {
                // row t of W (top) or Q~ into two 32-column TMA boxes (64 rows x 128 B, SW128: the
                // 16-byte chunk c of row t at c ^ (t % 8)); thread 0 stores the boxes after the
                // next barrier. W's boxes go to the A2 area, Q~'s to the Q halves of the input
                // tile and the upper R area (all read by no MMA any more).
                uint8_t* bx[2];
#pragma unroll
                for (int u = 0; u < 2; u++) bx[u] = top ? smem + C::kA2 + (2 * half + u) * 8192 : qt_box(2 * half + u);
                const float e = ex2_ftz(clt);  // e^{cl_t}, clt in log2 units
                const uint4* qrow = reinterpret_cast<const uint4*>(q + (row0 + t) * dk + 64 * half);
#pragma unroll
                for (int c8 = 0; c8 < 8; c8++) {
                    float w[8];
                    if (top) {
#pragma unroll
                        for (int e8 = 0; e8 < 8; e8++) w[e8] = v[8 * c8 + e8];
                    } else {
                        const uint4 u = qrow[c8];
                        const float2 f0 = unpack_bf16(u.x), f1 = unpack_bf16(u.y), f2 = unpack_bf16(u.z),
                                     f3 = unpack_bf16(u.w);
                        w[0] = e * (f0.x - v[8 * c8]); w[1] = e * (f0.y - v[8 * c8 + 1]);
                        w[2] = e * (f1.x - v[8 * c8 + 2]); w[3] = e * (f1.y - v[8 * c8 + 3]);
                        w[4] = e * (f2.x - v[8 * c8 + 4]); w[5] = e * (f2.y - v[8 * c8 + 5]);
                        w[6] = e * (f3.x - v[8 * c8 + 6]); w[7] = e * (f3.y - v[8 * c8 + 7]);
                    }
                    // floats 8 c8 .. 8 c8 + 7 of the row: box c8 / 4, chunks 2 (c8 % 4), 2 (c8 % 4) + 1
                    uint8_t* b = bx[c8 >> 2];
                    const int ch = 2 * (c8 & 3);
                    *reinterpret_cast<float4*>(b + t * 128 + ((ch ^ (t & 7)) << 4)) = make_float4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<float4*>(b + t * 128 + (((ch + 1) ^ (t & 7)) << 4)) =
                        make_float4(w[4], w[5], w[6], w[7]);
                }
            }
            tmem_ld32(tmem + lane_base + 192 + 32 * half, v);
            if (top) {
                // U row t scaled by its decay to the chunk end, bf16 hi + lo, MN-major rows of 64 dv
                const float w = ce[t];
                uint8_t* uh = smem + C::kR;
#pragma unroll
                for (int c8 = 0; c8 < 4; c8++) {
                    uint32_t h[4], l[4];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const float a = w * v[8 * c8 + 2 * e], b = w * v[8 * c8 + 2 * e + 1];
                        h[e] = pack_bf16(a, b);
                        const float2 hf = unpack_bf16(h[e]);
                        l[e] = pack_bf16(a - hf.x, b - hf.y);
                    }
                    *reinterpret_cast<uint4*>(uh + sw128_off(t, 4 * half + c8)) = make_uint4(h[0], h[1], h[2], h[3]);
                    *reinterpret_cast<uint4*>(uh + 8192 + sw128_off(t, 4 * half + c8)) =
                        make_uint4(l[0], l[1], l[2], l[3]);
                }
            } else if (N > 1) {
                // whole 64-byte runs of 8 rows per warp store (rows (t & ~3) + i of the lane group)
                float* dst = oacc + (row0 + (t & ~3)) * DV + 32 * half + 4 * (lane & 3);
#pragma unroll
                for (int hh = 0; hh < 2; hh++) {
                    uint4 y[4];
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const float* a = v + 16 * hh + 4 * j;
                        y[j] = make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                                          __float_as_uint(a[3]));
                    }
                    lane_group_transpose(y, lane);
#pragma unroll
                    for (int i = 0; i < 4; i++) *reinterpret_cast<uint4*>(dst + i * DV + 16 * hh) = y[i];
                }
            } else {
                uint4 y[4];
#pragma unroll
                for (int c8 = 0; c8 < 4; c8++)
                    y[c8] = make_uint4(pack_bf16(v[8 * c8], v[8 * c8 + 1]), pack_bf16(v[8 * c8 + 2], v[8 * c8 + 3]),
                                       pack_bf16(v[8 * c8 + 4], v[8 * c8 + 5]), pack_bf16(v[8 * c8 + 6], v[8 * c8 + 7]));
                lane_group_transpose(y, lane);
#pragma unroll
                for (int i = 0; i < 4; i++)
                    *reinterpret_cast<uint4*>(out + (row0 + (t & ~3) + i) * DV + 32 * half + 8 * (lane & 3)) = y[i];
            }
        }
        if (N == 1) break;
        fence_async_smem();
        block_sync();
        if (tid == 0) {
            // W and Q~ of the chunk: (dk / 32) boxes each
            const int wr = static_cast<int>((static_cast<size_t>(bh) * N + j) * C::kC);
            for (int b = 0; b < dk / 32; b++) {
                tma_store_2d(&tm_w, smem + C::kA2 + b * 8192, 32 * b, wr);
                tma_store_2d(&tm_qt, qt_box(b), 32 * b, wr);
            }
            bulk_commit();
            n_st = 1;
        }
        if (tid == 0) {
            const uint32_t kq = smem_u32(smem + C::kKQ), ub = smem_u32(smem + C::kR);
#pragma unroll
            for (int kk = 0; kk < 4; kk++)
#pragma unroll
                for (int h = 0; h < 2; h++)
                    mma_bf16(tmem, sdesc(kq + kk * 2048, C::kKQPanel, 1024), sdesc(ub + h * 8192 + kk * 2048, 8192, 1024),
                             idesc_bf16(128, 64, 1, 1), (kk > 0 || h > 0) ? 1u : 0u);
            mma_commit(mma_d);
            n_d = 1;
            wait(mma_d, 0);
            gam[static_cast<size_t>(bh) * N + j] = expf(cl[63]);
        }
        block_sync();
        if (*fail) break;
        {
            // the chunk's state: TMEM lane i = dk row i; warps 0..3 columns 0..31, warps 4..7 32..63
            const int c0 = 32 * (warp >> 2);
            float v[32];
            tmem_ld32(tmem + lane_base + c0, v);
            {
                // whole 64-byte runs of 8 rows per warp store; rows dk.. do not exist
                const int i0 = (warp & 3) * 32 + (lane & ~3);
                float* dst = nodes + (static_cast<size_t>(bh) * node_count + j) * static_cast<size_t>(dk) * DV +
                             static_cast<size_t>(i0) * DV + c0 + 4 * (lane & 3);
#pragma unroll
                for (int hh = 0; hh < 2; hh++) {
                    uint4 y[4];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const float* a = v + 16 * hh + 4 * e;
                        y[e] = make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                                          __float_as_uint(a[3]));
                    }
                    lane_group_transpose(y, lane);
#pragma unroll
                    for (int r = 0; r < 4; r++)
                        if (i0 + r < dk) *reinterpret_cast<uint4*>(dst + r * DV + 16 * hh) = y[r];
                }
            }
        }
    } while (false);

    if (tid == 0 && n_st) bulk_wait0();  // the stores of W and Q~ have read their boxes
    if (tid == 0 && *fail) {
        if (n_in) mbar_wait(in_full, 0);
        if (n_a) mbar_wait(mma_a, 0);
        if (n_bc) mbar_wait(mma_bc, 0);
        if (n_d) mbar_wait(mma_d, 0);
        if (n_m) mbar_wait(mma_m, 0);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace

bool gdn_level_tc_supported(const GdnPlan& pl, int dtype) {
    return dtype == 0 && pl.C == LvCfg::kC && pl.dv == LvCfg::kDV && (pl.dk == 64 || pl.dk == 128);
}

bool gdn_chunk_tc_supported(const GdnPlan& pl, int dtype) {
    return dtype == 0 && pl.C == CkCfg::kC && pl.dv == CkCfg::kDV && (pl.dk == 64 || pl.dk == 128);
}

// The chunk pass on tensor cores: W, Q~, node (0, j), gamma_j and the in-chunk output (into
// oacc, or straight into out when the sequence is one chunk).
cudaError_t gdn_chunk_tc(const GdnPlan& pl, const void* q, const void* k, const void* v, const float* log_a,
                         const float* beta, const float* lambda, float* Wg, float* Qt, float* nodes, float* gam,
                         float* oacc, void* out, int L, int* err, cudaStream_t stream) {
    const uint64_t rows = static_cast<uint64_t>(pl.B) * pl.H * pl.T;
    CUtensorMap tq, tk, tv, tw, tqt;
    const uint64_t wrows = static_cast<uint64_t>(pl.B) * pl.H * pl.N * CkCfg::kC;
    if (!make_map_box(&tq, q, false, rows, pl.dk, 64, CkCfg::kC) || !make_map_box(&tk, k, false, rows, pl.dk, 64, CkCfg::kC) ||
        !make_map_box(&tv, v, false, rows, pl.dv, 64, CkCfg::kC) ||
        !make_map_box(&tw, Wg, true, wrows, pl.dk, 32, CkCfg::kC) ||
        !make_map_box(&tqt, Qt, true, wrows, pl.dk, 32, CkCfg::kC))
        return cudaErrorInvalidValue;
    const int smem = CkCfg::kBytes + CkCfg::kSlack;
    cudaError_t e = cudaFuncSetAttribute(gdn_chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    gdn_chunk_tc_kernel<<<dim3(pl.N, pl.B * pl.H), 256, smem, stream>>>(
        tq, tk, tv, tw, tqt, static_cast<const __nv_bfloat16*>(q), log_a, beta, lambda, Wg, Qt, nodes, gam, oacc,
        static_cast<__nv_bfloat16*>(out), pl.T, pl.N, pl.dk, L, pl.node_count, err);
    note_launch(stream, "gdn_chunk_tc");
    return cudaGetLastError();
}

// All Fenwick levels of the prefill on tensor cores (one launch per level, in order).
cudaError_t gdn_levels_tc(const GdnPlan& pl, const void* k, const float* Wg, const float* Qt, float* nodes,
                          const float* gam, const float* lambda, float* oacc, int L, int c_log2, int* err,
                          cudaStream_t stream) {
    const uint64_t BH = static_cast<uint64_t>(pl.B) * pl.H;
    CUtensorMap tw, tq, tk;
    if (!make_map_box(&tw, Wg, true, BH * pl.N * LvCfg::kC, pl.dk, 32, LvCfg::kC) ||
        !make_map_box(&tq, Qt, true, BH * pl.N * LvCfg::kC, pl.dk, 32, LvCfg::kC) ||
        !make_map_box(&tk, k, false, BH * pl.T, pl.dk, 64, LvCfg::kC))
        return cudaErrorInvalidValue;
    const int smem = LvCfg::kBytes + LvCfg::kSlack;
    cudaError_t e = cudaFuncSetAttribute(gdn_level_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidValue;
    GdnTcLevels lo;
    for (int p = 0; p < 32; p++) lo.off[p] = pl.level_off[p];
    for (int p = 0; p < pl.P; p++) {
        const int n_even = (((pl.N - 1) >> p) + 1) / 2;
        if (n_even <= 0) continue;
        const int n_chains = static_cast<int>(BH) * n_even;
        const int grid = n_chains < 2 * sms ? n_chains : 2 * sms;
        gdn_level_tc_kernel<<<grid, 256, smem, stream>>>(tw, tq, tk, nodes, gam, lambda, oacc, pl.T, pl.N, pl.dk, L,
                                                         c_log2 + 1 + p, p, pl.P, pl.node_count, n_even, n_chains,
                                                         lo, err);
        note_launch(stream, "gdn_level_tc");
    }
    return cudaGetLastError();
}

}  // namespace lla
