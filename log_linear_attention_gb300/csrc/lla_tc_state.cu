// Tensor-core hand-off from prefill to decode: the Fenwick state set after a
// prompt of T tokens, for bf16 k/v with dk = 128 and dv in {64, 128}.
//
// After tokens 0..pos (pos = T - 1) the decode step holds, per head, one fp32
// dk x dv matrix per level l of pos's Fenwick walk ("Log-Linear Attention",
// pt §2 "Forma Recorrente e Paralela" / fr §2 "Algorithmes Efficaces": the
// finest bucket holds the newest token, coarser buckets are merged and
// promoted along the Fenwick tree):
//     slot l = sum over keys s at level l of exp(sum_{r=s+1..pos} log_a_r) k_s v_s^T,
// with level(pos, s) = 0 for s = pos, else 1 + floor(log2(pos xor s)).
// Slots whose level is empty for pos are left untouched.
//
// Layout on 128-token tiles (Pt = pos >> 7 full tiles precede the tile of pos):
//   * every key of a full tile u < Pt sits at level 8 + floor(log2(u xor Pt)),
//     so a full tile adds K_u^T diag(w) V_u to a single slot; the tiles of one
//     slot are consecutive;
//   * the keys of tile Pt (tokens 128 Pt .. pos) have levels 0..7.
// Kernels (one stream, in order):
//   state_tile_totals : g_u = sum of log_a over full tile u.
//   state_prep        : per head, (y = 0) tail_u = sum of log_a from the end of
//                       tile u to pos (reverse scan, newest first) and zeroes
//                       the slots >= 8 the next kernel adds into; (y = 1) the
//                       slots 0..7 from tile Pt, fp32 FMA.
//   tc_state          : persistent; each CTA takes an equal share of the
//                       flattened (head, full tile) list. Per tile,
//                       w_s = exp(tail_u + decay from s to the tile end), and
//                       w o V is split into bf16 hi + lo (so the product keeps
//                       ~16 mantissa bits); two tcgen05 MMAs per 16-token step
//                       accumulate K^T (w o V) in TMEM. A run of tiles of one
//                       slot ends with the accumulator added (fp32 vector
//                       atomics) into the slot.
// Every mbarrier wait is bounded; on overrun the kernel records LLA_ERR_TIMEOUT
// in the device error word, lets its own copies and MMAs land and returns.
#include "lla_tc_ptx.cuh"

namespace lla {
namespace {

constexpr int kPrepThreads = 256;
constexpr int kMaxStateTiles = 8192;  // a head's tile totals staged in shared memory

// grid (ceil(Pt / 8), BH), 256 threads: one warp per full tile.
__global__ void __launch_bounds__(256) state_tile_totals_kernel(const float* __restrict__ log_a,
                                                                float* __restrict__ g, int T, int Pt) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int u = blockIdx.x * 8 + warp, bh = blockIdx.y;
    if (u >= Pt) return;
    const float* a = log_a + static_cast<size_t>(bh) * T + static_cast<size_t>(u) * kTile;
    float s = a[lane] + a[lane + 32] + a[lane + 64] + a[lane + 96];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) g[static_cast<size_t>(bh) * Pt + u] = s;
}

// Exclusive prefix sum over the 256 threads of the block.
__device__ __forceinline__ float block_excl_scan256(float x, float* warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float incl = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    float base = 0.f;
    for (int w = 0; w < warp; w++) base += warp_tot[w];
    __syncthreads();
    return base + incl - x;
}

// grid (BH, 2), 256 threads, dynamic shared memory (see prep_smem_bytes).
template <int DV>
__global__ void __launch_bounds__(kPrepThreads)
    state_prep_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                      const float* __restrict__ log_a, const float* __restrict__ g, float* __restrict__ tail,
                      float* __restrict__ states, int T, int Pt, int Lmax) {
    extern __shared__ float psm[];
    __shared__ float warp_tot[8];
    __shared__ float la_sh[kTile];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int bh = blockIdx.x;
    const int pos = T - 1;
    const int base = Pt * kTile;     // first token of the tile of pos
    const int n = pos - base + 1;    // its tokens, 1..128
    const float* a = log_a + static_cast<size_t>(bh) * T;
    constexpr size_t msz = static_cast<size_t>(kDk) * DV;

    if (blockIdx.y == 0) {
        // tail_u for every full tile, summed from pos backwards
        float ts = (tid < n) ? a[base + tid] : 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ts += __shfl_xor_sync(0xffffffffu, ts, off);
        if (lane == 0) warp_tot[warp] = ts;
        __syncthreads();
        float tail_tot = 0.f;
        for (int w = 0; w < 8; w++) tail_tot += warp_tot[w];
        __syncthreads();
        float* g_sh = psm;
        for (int u = tid; u < Pt; u += kPrepThreads) g_sh[u] = g[static_cast<size_t>(bh) * Pt + u];
        __syncthreads();
        // thread t owns the tiles [hi - C, hi), hi = Pt - t C: thread 0 the newest
        const int C = (Pt + kPrepThreads - 1) / kPrepThreads;
        const int hi = Pt - tid * C;
        const int lo = hi - C > 0 ? hi - C : 0;
        float csum = 0.f;
        for (int u = hi - 1; u >= lo; u--) csum += g_sh[u];
        float run = tail_tot + block_excl_scan256(csum, warp_tot);
        for (int u = hi - 1; u >= lo; u--) {
            tail[static_cast<size_t>(bh) * Pt + u] = run;
            run += g_sh[u];
        }
        // zero the slots >= 8 held at pos (bit l - 8 of Pt): the MMA kernel adds into them
        float4* st4 = reinterpret_cast<float4*>(states + static_cast<size_t>(bh) * Lmax * msz);
        for (int l = 8; l < Lmax; l++) {
            if (((Pt >> (l - 8)) & 1) == 0) continue;
            for (size_t e = tid; e < msz / 4; e += kPrepThreads) st4[l * (msz / 4) + e] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        return;
    }

    // slots 0..7 from the tokens base .. pos: w_s = exp(sum_{r=s+1..pos} log_a_r)
    float* kw_sh = psm;                 // [128][kDk] fp32, w_s k_s
    float* v_sh = psm + kTile * kDk;    // [128][DV] fp32
    if (tid < kTile) la_sh[tid] = (tid < n) ? a[base + tid] : 0.f;
    __syncthreads();
    float suf = 0.f;  // summed from pos downwards
    if (tid < kTile)
        for (int r = n - 1; r > tid; r--) suf += la_sh[r];
    __syncthreads();
    if (tid < kTile) la_sh[tid] = suf;
    __syncthreads();
    const size_t row0 = static_cast<size_t>(bh) * T + base;
    for (int x = tid; x < n * kDk; x += kPrepThreads) {
        const int i = x / kDk, d = x % kDk;
        kw_sh[i * kDk + d] = expf(la_sh[i]) * __bfloat162float(k[(row0 + i) * kDk + d]);
    }
    for (int x = tid; x < n * DV; x += kPrepThreads) {
        const int i = x / DV, e = x % DV;
        v_sh[i * DV + e] = __bfloat162float(v[(row0 + i) * DV + e]);
    }
    __syncthreads();
    constexpr int EH = DV / 2;
    const int d = tid >> 1, e0 = (tid & 1) * EH;
    float acc[EH];
#pragma unroll
    for (int j = 0; j < EH; j++) acc[j] = 0.f;
    float* st = states + static_cast<size_t>(bh) * Lmax * msz + static_cast<size_t>(d) * DV + e0;
    int cur = fenwick_level(pos, base);
    for (int i = 0; i < n; i++) {
        const int l = fenwick_level(pos, base + i);
        if (l != cur) {
            float4* dst = reinterpret_cast<float4*>(st + cur * msz);
#pragma unroll
            for (int j = 0; j < EH / 4; j++) dst[j] = make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
#pragma unroll
            for (int j = 0; j < EH; j++) acc[j] = 0.f;
            cur = l;
        }
        const float kd = kw_sh[i * kDk + d];
        const float4* vr = reinterpret_cast<const float4*>(v_sh + i * DV + e0);
#pragma unroll
        for (int j = 0; j < EH / 4; j++) {
            const float4 x = vr[j];
            acc[4 * j] = fmaf(kd, x.x, acc[4 * j]);
            acc[4 * j + 1] = fmaf(kd, x.y, acc[4 * j + 1]);
            acc[4 * j + 2] = fmaf(kd, x.z, acc[4 * j + 2]);
            acc[4 * j + 3] = fmaf(kd, x.w, acc[4 * j + 3]);
        }
    }
    float4* dst = reinterpret_cast<float4*>(st + cur * msz);
#pragma unroll
    for (int j = 0; j < EH / 4; j++) dst[j] = make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
}

template <int DV>
size_t prep_smem_bytes(int Pt) {
    const size_t tiles = static_cast<size_t>(kTile) * (kDk + DV) * sizeof(float);
    const size_t scan = static_cast<size_t>(Pt) * sizeof(float);
    return tiles > scan ? tiles : scan;
}

template <int DV>
struct StateCfg {
    static constexpr int kStages = DV == 64 ? 3 : 2;
    static constexpr int kKBytes = 2 * kPanelBytes;            // K tile: 128 tokens x 128 dk
    static constexpr int kVBytes = (DV / 64) * kPanelBytes;    // V tile (scaled hi in place) / the lo part
    static constexpr int kStageBytes = kKBytes + 2 * kVBytes;
    static constexpr uint32_t kTxBytes = kKBytes + kVBytes;
    static constexpr int kBytes = kStages * kStageBytes + 1024;  // + alignment slack
    static constexpr int kThreads = 384;
    static constexpr uint32_t kTmemCols = 2 * DV;              // two accumulators
};

// Level of full tile u (< Pt) for the last token pos (Pt = pos >> 7).
__device__ __forceinline__ int tile_level(int u, int Pt) { return 8 + 31 - __clz(u ^ Pt); }

// 384 threads: warp 0 TMA producer, warp 1 TMEM owner + MMA issuer, warps 4..7
// scale V (one token row per thread), warps 8..11 drain accumulators (TMEM lane
// quadrant = warp % 4, one dk row per thread).
template <int DV>
__global__ void __launch_bounds__(384, 1)
    tc_state_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const float* __restrict__ log_a, const float* __restrict__ tail, float* __restrict__ states,
                    int T, int Pt, int Lmax, int total, int* err) {
    using C = StateCfg<DV>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full_bar[S], scaled_bar[S], empty_bar[S], acc_full[2], acc_empty[2], drain_bar;
    __shared__ uint32_t tmem_base_sh;
    __shared__ float wt_sh[2][4];
    __shared__ int fail_sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * total / gridDim.x);
    const int t1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * total / gridDim.x);
    volatile int* fail = &fail_sh;

    if (tid == 0) {
        for (int s = 0; s < S; s++) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&scaled_bar[s], 4);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        mbar_init(&drain_bar, 1);
        fence_mbar_init();
        fail_sh = 0;
    }
    if (warp == 1) tmem_alloc(&tmem_base_sh, C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    auto fail_now = [&]() {
        if (atomicExch(&fail_sh, 1) == 0) record_error(err, kDevTimeout);
    };
    // same slot for flattened tiles f and f + 1
    auto same_run = [&](int f) {
        const int b0 = f / Pt, b1 = (f + 1) / Pt;
        return b0 == b1 && tile_level(f % Pt, Pt) == tile_level((f + 1) % Pt, Pt);
    };

    int issued = 0;  // producer: tiles whose copies were issued
    if (warp == 0) {
        if (lane == 0) {
            for (int f = t0; f < t1 && !*fail; f++, issued++) {
                const int i = f - t0, s = i % S;
                if (i >= S && !mbar_wait(&empty_bar[s], ((i / S) - 1) & 1)) {
                    fail_now();
                    break;
                }
                const int bh = f / Pt, u = f % Pt;
                const int r0 = bh * T + u * kTile;
                uint8_t* st = smem + s * C::kStageBytes;
                mbar_expect_tx(&full_bar[s], C::kTxBytes);
                tma_load_2d(st, &tm_k, &full_bar[s], 0, r0);
                tma_load_2d(st + kPanelBytes, &tm_k, &full_bar[s], 64, r0);
#pragma unroll
                for (int p = 0; p < DV / 64; p++)
                    tma_load_2d(st + C::kKBytes + p * kPanelBytes, &tm_v, &full_bar[s], 64 * p, r0);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t kIdesc = idesc_bf16(kDk, DV, 1, 1);  // A = K^T (MN-major), B = w o V (MN-major)
            int run = 0;
            for (int f = t0; f < t1 && !*fail; f++) {
                const int i = f - t0, s = i % S;
                const bool starting = (f == t0) || !same_run(f - 1);
                const bool ending = (f == t1 - 1) || !same_run(f);
                const int buf = run & 1;
                if (starting && run >= 2 && !mbar_wait(&acc_empty[buf], ((run >> 1) - 1) & 1)) {
                    fail_now();
                    break;
                }
                if (!mbar_wait(&scaled_bar[s], (i / S) & 1)) {
                    fail_now();
                    break;
                }
                tc_fence_after();
                const uint32_t kb = smem_u32(smem + s * C::kStageBytes);
                const uint32_t vb = kb + C::kKBytes, lb = vb + C::kVBytes;
                const uint32_t d = tmem + buf * DV;
#pragma unroll
                for (int kk = 0; kk < kTile / 16; kk++) {
                    const uint64_t ad = sdesc(kb + kk * 2048, kPanelBytes, 1024);
                    mma_bf16(d, ad, sdesc(vb + kk * 2048, kPanelBytes, 1024), kIdesc, (starting && kk == 0) ? 0u : 1u);
                    mma_bf16(d, ad, sdesc(lb + kk * 2048, kPanelBytes, 1024), kIdesc, 1u);
                }
                mma_commit(&empty_bar[s]);
                if (ending) {
                    mma_commit(&acc_full[buf]);
                    run++;
                }
            }
            // every MMA issued above has completed before TMEM and shared memory go away
            mma_commit(&drain_bar);
            if (!mbar_wait(&drain_bar, 0)) fail_now();
        }
    } else if (warp >= 4 && warp < 8) {
        const int row = tid - 128, w4 = warp - 4;
        float la_next = 0.f, tail_next = 0.f;
        if (t0 < t1) {
            la_next = log_a[static_cast<size_t>(t0 / Pt) * T + (t0 % Pt) * kTile + row];
            tail_next = tail[t0];
        }
        for (int f = t0; f < t1; f++) {
            const int i = f - t0, s = i % S;
            const float la = la_next, tl = tail_next;
            if (f + 1 < t1) {
                la_next = log_a[static_cast<size_t>((f + 1) / Pt) * T + ((f + 1) % Pt) * kTile + row];
                tail_next = tail[f + 1];
            }
            // decay from token row to the tile end: total - inclusive prefix
            float incl = la;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            if (lane == 31) wt_sh[i & 1][w4] = incl;
            // the four scaler warps meet here each tile and leave together on a failure
            uint32_t stop;
            asm volatile(
                "{\n\t.reg .pred p, q;\n\t"
                "setp.ne.b32 q, %1, 0;\n\t"
                "bar.red.or.pred p, 1, 128, q;\n\t"
                "selp.u32 %0, 1, 0, p;\n\t}"
                : "=r"(stop)
                : "r"(*fail)
                : "memory");
            if (stop) break;
            float before = 0.f, tot = 0.f;
#pragma unroll
            for (int w = 0; w < 4; w++) {
                const float x = wt_sh[i & 1][w];
                before += (w < w4) ? x : 0.f;
                tot += x;
            }
            const float w = exp2f((tl + tot - (before + incl)) * kLog2e);
            if (!warp_wait(&full_bar[s], (i / S) & 1)) {
                if (lane == 0) fail_now();
                continue;  // the next meeting sees the failure
            }
            uint8_t* vrow = smem + s * C::kStageBytes + C::kKBytes + row * 128;
#pragma unroll
            for (int p = 0; p < DV / 64; p++) {
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    const uint32_t off = p * kPanelBytes + ((c ^ (row & 7)) << 4);
                    uint4* hp = reinterpret_cast<uint4*>(vrow + off);
                    uint4* lp = reinterpret_cast<uint4*>(vrow + C::kVBytes + off);
                    const uint4 x = *hp;
                    const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
                    uint32_t hs[4], ls[4];
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const float2 f2 = unpack_bf16(xs[q]);
                        const float a0 = f2.x * w, a1 = f2.y * w;
                        hs[q] = pack_bf16(a0, a1);
                        const float2 h2 = unpack_bf16(hs[q]);
                        ls[q] = pack_bf16(a0 - h2.x, a1 - h2.y);
                    }
                    *hp = make_uint4(hs[0], hs[1], hs[2], hs[3]);
                    *lp = make_uint4(ls[0], ls[1], ls[2], ls[3]);
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&scaled_bar[s]);
        }
    } else if (warp >= 8) {
        const int quad = warp & 3;
        const int d = quad * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        int run = 0;
        for (int f = t0; f < t1; f++) {
            if (!((f == t1 - 1) || !same_run(f))) continue;
            const int buf = run & 1;
            if (*fail) break;
            if (!warp_wait(&acc_full[buf], (run >> 1) & 1)) {
                if (lane == 0) fail_now();
                break;
            }
            tc_fence_after();
            const int bh = f / Pt, l = tile_level(f % Pt, Pt);
            float4* dst = reinterpret_cast<float4*>(states + ((static_cast<size_t>(bh) * Lmax + l) * kDk + d) * DV);
#pragma unroll
            for (int c0 = 0; c0 < DV; c0 += 32) {
                float x[32];
                tmem_ld32(tmem + lane_base + buf * DV + c0, x);
#pragma unroll
                for (int j = 0; j < 8; j++)
                    atomicAdd(dst + c0 / 4 + j, make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
            run++;
        }
    }

    __syncthreads();
    if (*fail && warp == 0 && lane == 0) {
        // let the copies still in flight land before the shared memory goes away
        for (int i = issued - S > 0 ? issued - S : 0; i < issued; i++) mbar_wait(&full_bar[i % S], (i / S) & 1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

template <int DV>
cudaError_t tc_prefill_state_dv(const void* k, const void* v, const float* log_a, float* states, int BH, int T,
                                int Lmax, void* workspace, int* err, cudaStream_t stream) {
    const int pos = T - 1;
    const int Pt = pos >> 7;
    float* g = static_cast<float*>(workspace);
    float* tail = g + static_cast<size_t>(BH) * Pt;
    if (Pt > 0) {
        state_tile_totals_kernel<<<dim3((Pt + 7) / 8, BH), 256, 0, stream>>>(log_a, g, T, Pt);
        note_launch(stream, "state_tile_totals");
    }
    {
        const size_t smem = prep_smem_bytes<DV>(Pt);
        cudaError_t e = cudaFuncSetAttribute(state_prep_kernel<DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        state_prep_kernel<DV><<<dim3(BH, 2), kPrepThreads, smem, stream>>>(
            static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), log_a, g, tail, states, T,
            Pt, Lmax);
        note_launch(stream, "state_prep");
    }
    if (Pt > 0) {
        CUtensorMap tk, tv;
        const uint64_t rows = static_cast<uint64_t>(BH) * T;
        if (!make_map(&tk, k, rows, kDk) || !make_map(&tv, v, rows, DV)) return cudaErrorInvalidValue;
        using C = StateCfg<DV>;
        cudaError_t e = cudaFuncSetAttribute(tc_state_kernel<DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kBytes);
        if (e != cudaSuccess) return e;
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
            cudaGetLastError();
            sms = 152;
        }
        const int total = BH * Pt;
        const int grid = total < sms ? total : sms;
        tc_state_kernel<DV><<<grid, C::kThreads, C::kBytes, stream>>>(tk, tv, log_a, tail, states, T, Pt, Lmax,
                                                                       total, err);
        note_launch(stream, "tc_state");
    }
    return cudaGetLastError();
}

}  // namespace

bool tc_state_supported(int dtype, int dk, int dv, int B, int H, int T) {
    const int64_t Pt = (static_cast<int64_t>(T) - 1) >> 7;
    return dtype == 0 && dk == kDk && (dv == 64 || dv == 128) && Pt <= kMaxStateTiles &&
           static_cast<int64_t>(B) * H * T < (int64_t(1) << 31);
}

size_t tc_state_workspace_bytes(int B, int H, int T) {
    return 2 * static_cast<size_t>(B) * H * (static_cast<size_t>(T - 1) >> 7) * sizeof(float) + 256;
}

cudaError_t tc_prefill_state(const void* k, const void* v, const float* log_a, float* states, int B, int H, int T,
                             int dv, int Lmax, void* workspace, int* err, cudaStream_t stream) {
    if (dv == 64) return tc_prefill_state_dv<64>(k, v, log_a, states, B * H, T, Lmax, workspace, err, stream);
    return tc_prefill_state_dv<128>(k, v, log_a, states, B * H, T, Lmax, workspace, err, stream);
}

}  // namespace lla
