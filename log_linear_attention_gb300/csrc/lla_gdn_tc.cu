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

// grid (number of read nodes of level p per head, B*H), 128 threads (thread = TMEM lane),
// two CTAs per SM.
__global__ void __launch_bounds__(128, 2)
    gdn_level_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_qt,
                        const __grid_constant__ CUtensorMap tm_k, float* __restrict__ nodes,
                        const float* __restrict__ gam, const float* __restrict__ lambda, float* __restrict__ oacc,
                        int T, int N, int dk, int L, int lev, int p, int P, int node_count,
                        const __grid_constant__ GdnTcLevels lo, int* err) {
    using C = LvCfg;
    constexpr int DV = C::kDV;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    uint64_t* full_a = reinterpret_cast<uint64_t*>(smem + C::kBar);
    uint64_t* full_k = full_a + 1;
    uint64_t* mma1 = full_a + 2;
    uint64_t* mma2 = full_a + 3;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full_a + 4);
    volatile int* fail = reinterpret_cast<volatile int*>(full_a + 5);

    const int tid = threadIdx.x, warp = tid >> 5;
    if (pad > static_cast<uint32_t>(C::kSlack)) {  // base alignment below the assumed 128 bytes
        if (tid == 0) record_error(err, kDevBadInput);
        return;
    }
    const int xi = blockIdx.x, bh = blockIdx.y;
    const int m = 2 * xi, span = 1 << p;
    const int b0 = (m + 1) * span, b1 = min((m + 2) * span, N);
    const bool want_parent = (m + 2) * span <= N && p + 1 < P;
    const size_t msz = static_cast<size_t>(dk) * DV;

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
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tD = tmem + lane_base;       // MMA1 result, columns [0, 64)
    const uint32_t tX = tmem + lane_base + 64;  // carried node, columns [64, 128)
    constexpr uint32_t kIdA = idesc_tf32(128, DV);        // [W; Q~] (K-major) x X (K-major)
    constexpr uint32_t kIdB = idesc_bf16(128, DV, 1, 1);  // K^T (MN-major) x Y (MN-major)

    int n_a = 0, n_k = 0, n_m1 = 0, n_m2 = 0;  // copies and MMA groups issued (thread 0)
    auto load_a = [&](int jc) {
        const int r = (bh * N + jc) * C::kC;
        mbar_expect_tx(full_a, C::kABytes);
#pragma unroll
        for (int q = 0; q < 4; q++) {
            tma_load_2d(smem + C::kA + q * C::kAPanel, &tm_w, full_a, 32 * q, r);
            tma_load_2d(smem + C::kA + q * C::kAPanel + C::kAPanel / 2, &tm_qt, full_a, 32 * q, r);
        }
        n_a++;
    };
    auto load_k = [&](int jc) {
        const int r = bh * T + jc * C::kC;
        mbar_expect_tx(full_k, C::kKBytes);
        tma_load_2d(smem + C::kK, &tm_k, full_k, 0, r);
        tma_load_2d(smem + C::kK + C::kKPanel, &tm_k, full_k, 64, r);
        n_k++;
    };
    // thread 0 waits; the block learns the outcome from `fail` after its next barrier
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (mbar_wait(bar, parity)) return true;
        *fail = 1;
        record_error(err, kDevTimeout);
        return false;
    };
    // X row i (i = tid, a dk row) into the K-major fp32 staging of X^T: element (d, i) sits in
    // panel i / 32, row d, 16-byte chunk ((i % 32) / 4) ^ (d % 8), word i % 4
    auto stage_xt = [&](const float* x) {
        uint8_t* base = smem + C::kX + (tid >> 5) * C::kXPanel + (tid & 3) * 4;
        const int c = (tid & 31) >> 2;
#pragma unroll
        for (int d = 0; d < DV; d++) *reinterpret_cast<float*>(base + d * 128 + ((c ^ (d & 7)) << 4)) = x[d];
    };

    if (tid == 0) {
        load_a(b0);
        load_k(b0);
    }
    {
        // X = node (p, m); rows dk..127 are zero
        float x[DV];
        const float4* src = reinterpret_cast<const float4*>(
            nodes + (static_cast<size_t>(bh) * node_count + lo.off[p] + m) * msz + static_cast<size_t>(tid) * DV);
#pragma unroll
        for (int c4 = 0; c4 < DV / 4; c4++) {
            const float4 f = tid < dk ? src[c4] : make_float4(0.f, 0.f, 0.f, 0.f);
            x[4 * c4] = f.x; x[4 * c4 + 1] = f.y; x[4 * c4 + 2] = f.z; x[4 * c4 + 3] = f.w;
        }
        tmem_st32(tX, x);
        tmem_st32(tX + 32, x + 32);
        stage_xt(x);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    float Gam = 1.f;  // product of gamma over the chunks passed
    for (int jc = b0, s = 0; jc < b1; jc++, s++) {
        const uint32_t ph = s & 1;
        const bool last = jc + 1 == b1;
        const bool carry = !last || want_parent;
        if (tid == 0 && wait(full_a, ph)) {
            tc_fence_after();
            const uint32_t ab = smem_u32(smem + C::kA), xb = smem_u32(smem + C::kX);
#pragma unroll
            for (int kk = 0; kk < 16; kk++) {
                const uint32_t oa = (kk >> 2) * C::kAPanel + (kk & 3) * 32;
                const uint32_t ob = (kk >> 2) * C::kXPanel + (kk & 3) * 32;
                mma_tf32(tmem, sdesc(ab + oa, 16, 1024), sdesc(xb + ob, 16, 1024), kIdA, kk > 0 ? 1u : 0u);
            }
            mma_commit(mma1);
            n_m1++;
            if (wait(mma1, ph) && !last) load_a(jc + 1);  // MMA1 has read the stage
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (*fail) break;
        const size_t row0 = static_cast<size_t>(bh) * T + static_cast<size_t>(jc) * C::kC;
        float v[DV];
        tmem_ld32(tD, v);
        tmem_ld32(tD + 32, v + 32);
        if (tid < C::kC) {
            if (carry) {
                // -Y row tid as bf16 hi + lo, MN-major rows of 64 dv (one 128-byte row per token)
                uint8_t* hi = smem + C::kX;
                uint8_t* lo_ = smem + C::kX + C::kXPanel;
#pragma unroll
                for (int c8 = 0; c8 < DV / 8; c8++) {
                    uint32_t h[4], l[4];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const float a = -v[8 * c8 + 2 * e], b = -v[8 * c8 + 2 * e + 1];
                        h[e] = pack_bf16(a, b);
                        const float2 hf = unpack_bf16(h[e]);
                        l[e] = pack_bf16(a - hf.x, b - hf.y);
                    }
                    *reinterpret_cast<uint4*>(hi + sw128_off(tid, c8)) = make_uint4(h[0], h[1], h[2], h[3]);
                    *reinterpret_cast<uint4*>(lo_ + sw128_off(tid, c8)) = make_uint4(l[0], l[1], l[2], l[3]);
                }
            }
        } else {
            const size_t t = row0 + (tid - C::kC);
            const float w = lambda[t * L + lev] * Gam;
            float4* o = reinterpret_cast<float4*>(oacc + t * DV);
#pragma unroll
            for (int c4 = 0; c4 < DV / 4; c4++) {
                float4 a = o[c4];
                a.x = fmaf(w, v[4 * c4], a.x);
                a.y = fmaf(w, v[4 * c4 + 1], a.y);
                a.z = fmaf(w, v[4 * c4 + 2], a.z);
                a.w = fmaf(w, v[4 * c4 + 3], a.w);
                o[c4] = a;
            }
        }
        if (!carry) break;
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
            if (wait(mma2, ph) && !last) load_k(jc + 1);  // MMA2 has read K
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (*fail) break;
        Gam *= gam[static_cast<size_t>(bh) * N + jc];
        tmem_ld32(tX, v);
        tmem_ld32(tX + 32, v + 32);
        if (!last) {
            stage_xt(v);
        } else if (tid < dk) {
            // node (p + 1, m / 2) = Gamma X^ + node (p, m + 1)
            const float4* sib = reinterpret_cast<const float4*>(
                nodes + (static_cast<size_t>(bh) * node_count + lo.off[p] + m + 1) * msz + static_cast<size_t>(tid) * DV);
            float4* dst = reinterpret_cast<float4*>(
                nodes + (static_cast<size_t>(bh) * node_count + lo.off[p + 1] + xi) * msz + static_cast<size_t>(tid) * DV);
#pragma unroll
            for (int c4 = 0; c4 < DV / 4; c4++) {
                const float4 b = sib[c4];
                dst[c4] = make_float4(fmaf(Gam, v[4 * c4], b.x), fmaf(Gam, v[4 * c4 + 1], b.y),
                                      fmaf(Gam, v[4 * c4 + 2], b.z), fmaf(Gam, v[4 * c4 + 3], b.w));
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
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

}  // namespace

bool gdn_level_tc_supported(const GdnPlan& pl, int dtype) {
    return dtype == 0 && pl.C == LvCfg::kC && pl.dv == LvCfg::kDV && (pl.dk == 64 || pl.dk == 128);
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
    GdnTcLevels lo;
    for (int p = 0; p < 32; p++) lo.off[p] = pl.level_off[p];
    for (int p = 0; p < pl.P; p++) {
        const int n_even = (((pl.N - 1) >> p) + 1) / 2;
        if (n_even <= 0) continue;
        gdn_level_tc_kernel<<<dim3(n_even, static_cast<unsigned>(BH)), 128, smem, stream>>>(
            tw, tq, tk, nodes, gam, lambda, oacc, pl.T, pl.N, pl.dk, L, c_log2 + 1 + p, p, pl.P, pl.node_count, lo,
            err);
        note_launch(stream, "gdn_level_tc");
    }
    return cudaGetLastError();
}

}  // namespace lla
