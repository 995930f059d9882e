// Tensor-core (tcgen05 / TMEM / TMA) backward of log-linear Mamba-2 attention
// for bf16 q/k/v/dO with dk = 128, dv = 64 and T % 128 == 0.
//
// The gradients of L = sum_t dO_t . o_t follow the forward's structure on
// 128-token tiles ("Log-Linear Attention", pt §2 "Forma Recorrente e Paralela"
// / fr §2 "Algorithmes Efficaces": dense work inside a block, Fenwick nodes
// across blocks). Tile j reads node (p, m = (j >> p) - 1) for each set bit p of
// j with per-query weight r_{t,p} = lambda_t^(8+p) exp(cum_t - cum_e), e the
// node's last token; inside a tile the key levels are 0..7.
//
// Kernels (one stream, in order):
//   tc_nodes, tc_merge : the forward's node stage (bf16 nodes that are read,
//                        tile decays, per-token and per-level decay tables).
//   tc_dnode_zero_cut  : zeroes the nodes whose reading block a CTA boundary of
//                        tc_dnode cuts.
//   tc_dnode           : node gradients dB_{p,m} = sum over the tiles j of the
//                        reading block of Q_j^T diag(r_p) dO_j, on tcgen05 with
//                        r_p o dO scaled in shared memory; tile-major (Q, dO
//                        read once per tile), each level's run accumulates in
//                        its TMEM slot and leaves by a TMA store (a whole run)
//                        or TMA reduce-adds (a run cut by a CTA boundary).
//   tc_cmat            : per key tile i, C_i = sum over its read ancestor
//                        nodes of exp(decay from tile i's end to the node's
//                        end) dB (bf16, an MMA operand of the next kernel).
//   tc_bwd_tile        : persistent, one CTA per SM and one (head, tile) item at
//                        a time: S = Q K^T and dP = dO V^T (TMEM), and beside
//                        the epilogue the key side, dK = (w o V) C_i^T and
//                        Z = K C_i (for dcum and dV's term diag(w) Z);
//                        A = lambda D S and G = lambda D dP (bf16, smem) with
//                        dlambda levels 0..7 and the decay derivatives; then
//                        dV = A^T dO, dQ = G K, dK += G^T Q; per set bit p (two
//                        at a time), Y_p = Q B_p (for dlambda_t^(8+p) and dcum)
//                        and dQ += (r_p o dO) B_p^T; dQ, dK, dV leave by TMA
//                        stores while the next item's inputs are copied in.
//   bwd_dloga          : dlog_a_r = sum_{t >= r} dcum_t.
// Every mbarrier wait is bounded; on overrun a kernel records LLA_ERR_TIMEOUT,
// lets its own copies and MMAs land and returns.
#include "lla_tc_ptx.cuh"

namespace lla {
namespace {

constexpr int kDV = 64;
constexpr int kMsz = kDk * kDV;

struct Offsets { int off[32]; };

// ------------------------------------------------------------------ tc_dnode

// Tile-major: the CTA walks an equal share of the (head, tile) list; each tile's Q and dO
// are loaded once, and for every set bit p of the tile index in the pass's level window
// [p_lo, p_lo + np) the scaler warps write r_p o dO into a slot of the scaled ring. Level
// p accumulates in TMEM columns 64 (p - p_lo) over the tiles of its reading block (a run)
// and is drained into its node when the run ends: at the block's last tile, at the
// head's last tile or at the end of the CTA's share. A drain warp stages its 32 rows in
// shared memory and adds them to the fp32 node with TMA reduce-adds in L2 (partial runs of
// neighbouring CTAs meet there).
struct DnodeCfg {
    static constexpr int kRaw = 2;                               // Q + dO stages
    static constexpr int kScaled = 4;                            // r_p o dO slots
    static constexpr int kQBytes = 2 * kPanelBytes;              // Q tile: 128 tokens x 128
    static constexpr int kRawBytes = kQBytes + kPanelBytes;      // + dO tile: 128 tokens x 64
    static constexpr int kDrainBytes = 2 * 4096;                 // per drain warp: 32 rows x 64 fp32
    static constexpr int kBytes = kRaw * kRawBytes + kScaled * kPanelBytes + 4 * kDrainBytes + 1024;
    static constexpr int kThreads = 384;
    static constexpr int kMaxLevels = 8;                         // 8 x 64 TMEM columns
    // dynamic + the kernel's static arrays (w_sh, barriers) within the 227 KB a CTA may hold
    static_assert(kBytes + kMaxLevels * kTile * 4 + 512 <= 227 * 1024, "tc_dnode shared memory");
};

// Level window of one tile: bit q of `bits` = level p_lo + q is read by the tile; `start` /
// `end` mark the levels whose run this CTA begins / finishes at the tile; `start_cut` /
// `end_cut` the subset where that is only because the CTA's share begins / ends there (the
// run continues in a neighbouring CTA).
struct DnodeTile {
    int bh, j;
    uint32_t bits, start, end, start_cut, end_cut;
};

// Tile f of the flattened (head, tile) list is tile j of head bh (the callers step both along f).
__device__ __forceinline__ DnodeTile dnode_tile(int f, int bh, int j, int NT, int p_lo, int np, int t0, int t1) {
    DnodeTile d;
    d.bh = bh;
    d.j = j;
    d.bits = (static_cast<uint32_t>(d.j) >> p_lo) & ((1u << np) - 1u);
    d.start = d.end = d.start_cut = d.end_cut = 0;
#pragma unroll
    for (int q = 0; q < DnodeCfg::kMaxLevels; q++) {
        if (!((d.bits >> q) & 1u)) continue;
        const int full = (1 << (p_lo + q)) - 1, low = d.j & full;
        const bool natural_end = low == full || d.j + 1 == NT;
        if (f == t0 || low == 0) d.start |= 1u << q;
        if (natural_end || f + 1 == t1) d.end |= 1u << q;
        if (low != 0 && f == t0) d.start_cut |= 1u << q;
        if (!natural_end && f + 1 == t1) d.end_cut |= 1u << q;
    }
    return d;
}

// 384 threads: warp 0 TMA producer, warp 1 TMEM owner + MMA issuer, warps 4..7 scale
// dO (one token row per thread), warps 8..11 drain accumulators (dk row per thread).
__global__ void __launch_bounds__(384, 1)
    tc_dnode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dn, const float* __restrict__ lambda, const float* __restrict__ tok_cl2,
                    const float* __restrict__ dtab, int T, int NT, int L, int node_count,
                    const __grid_constant__ Offsets lo, int p_lo, int np, int total, int* err) {
    using C = DnodeCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* scaled = smem + C::kRaw * C::kRawBytes;
    uint8_t* drain_stage = scaled + C::kScaled * kPanelBytes;
    __shared__ uint64_t raw_full[C::kRaw], raw_empty[C::kRaw], sc_full[C::kScaled], sc_empty[C::kScaled];
    __shared__ uint64_t acc_full[C::kMaxLevels], acc_empty[C::kMaxLevels], drain_bar;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int fail_sh;
    __shared__ int lo_sh[32];
    __shared__ float w_sh[DnodeCfg::kMaxLevels][kTile];  // this tile's r_{t, p_lo + q}, row t written by its scaler

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * total / gridDim.x);
    const int t1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * total / gridDim.x);
    const uint32_t tmem_cols = np <= 2 ? 128u : (np <= 4 ? 256u : 512u);
    volatile int* fail = &fail_sh;
    if (tid < 32) lo_sh[tid] = lo.off[tid];

    if (tid == 0) {
        for (int s = 0; s < C::kRaw; s++) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], 1);
        }
        for (int s = 0; s < C::kScaled; s++) {
            mbar_init(&sc_full[s], 4);
            mbar_init(&sc_empty[s], 1);
        }
        for (int q = 0; q < C::kMaxLevels; q++) {
            mbar_init(&acc_full[q], 1);
            mbar_init(&acc_empty[q], 4);
        }
        mbar_init(&drain_bar, 1);
        fence_mbar_init();
        fail_sh = 0;
    }
    if (warp == 1) tmem_alloc(&tmem_base_sh, tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    auto fail_now = [&]() {
        if (atomicExch(&fail_sh, 1) == 0) record_error(err, kDevTimeout);
    };
    // the window's level bits of tile j of a head; the loops below step (head, j) along the
    // flattened tile index f instead of dividing it
    auto lbits = [&](int j) { return (static_cast<uint32_t>(j) >> p_lo) & ((1u << np) - 1u); };
    auto step = [&](int& j, int& bh) {
        if (++j == NT) {
            j = 0;
            bh++;
        }
    };
    const int bh0 = t0 / NT, j0 = t0 - (t0 / NT) * NT;

    int issued = 0;
    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int j = j0, bh = bh0;
            for (int f = t0; f < t1 && !*fail; f++, step(j, bh)) {
                if (lbits(j) == 0) continue;
                if (issued >= C::kRaw && !mbar_wait(&raw_empty[s], ph ^ 1u)) {
                    fail_now();
                    break;
                }
                const int r0 = f * kTile;  // (bh * NT + j) * 128 = bh * T + 128 j
                uint8_t* st = smem + s * C::kRawBytes;
                mbar_expect_tx(&raw_full[s], C::kRawBytes);
                tma_load_2d(st, &tm_q, &raw_full[s], 0, r0);
                tma_load_2d(st + kPanelBytes, &tm_q, &raw_full[s], 64, r0);
                tma_load_2d(st + C::kQBytes, &tm_do, &raw_full[s], 0, r0);
                issued++;
                if (++s == C::kRaw) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t kIdesc = idesc_bf16(kDk, kDV, 1, 1);  // A = Q^T, B = r o dO, both MN-major
            const uint64_t qdesc0 = sdesc(smem_u32(smem), kPanelBytes, 1024);
            const uint64_t ddesc0 = sdesc(smem_u32(scaled), kPanelBytes, 1024);
            constexpr uint64_t kRawStep = C::kRawBytes >> 4, kScStep = kPanelBytes >> 4;
            int rs = 0, ss = 0;
            uint32_t sph = 0, run_par = 0, used = 0;
            int j = j0, bh = bh0;
            for (int f = t0; f < t1 && !*fail; f++, step(j, bh)) {
                const DnodeTile d = dnode_tile(f, bh, j, NT, p_lo, np, t0, t1);
                if (d.bits == 0) continue;
                bool ok = true;
#pragma unroll 1
                for (uint32_t b = d.bits; b != 0; b &= b - 1) {
                    const int q = __ffs(b) - 1;
                    const bool st = (d.start >> q) & 1u;
                    if (st) {
                        if (((used >> q) & 1u) && !mbar_wait(&acc_empty[q], ((run_par >> q) & 1u) ^ 1u)) {
                            ok = false;
                            break;
                        }
                        used |= 1u << q;
                        run_par ^= 1u << q;
                    }
                    if (!mbar_wait(&sc_full[ss], sph)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; kk++) {
                        const uint64_t ko = 128u * kk;
                        mma_bf16(tmem + q * kDV, qdesc0 + kRawStep * rs + ko, ddesc0 + kScStep * ss + ko, kIdesc,
                                 (st && kk == 0) ? 0u : 1u);
                    }
                    mma_commit(&sc_empty[ss]);
                    if ((d.end >> q) & 1u) mma_commit(&acc_full[q]);
                    if (++ss == C::kScaled) {
                        ss = 0;
                        sph ^= 1u;
                    }
                }
                if (!ok) {
                    fail_now();
                    break;
                }
                mma_commit(&raw_empty[rs]);
                if (++rs == C::kRaw) rs = 0;
            }
            mma_commit(&drain_bar);
            if (!mbar_wait(&drain_bar, 0)) fail_now();
        }
    } else if (warp >= 4 && warp < 8) {
        const int row = tid - 128;
        // r_{t,p} = lambda_t^(8+p) exp2(cl2_t + dtab[j][p]) for this thread's token row; the
        // factors of the next tile are fetched while the current one is scaled.
        float lam[C::kMaxLevels], dt[C::kMaxLevels], cl2 = 0.f;
        float nlam[C::kMaxLevels], ndt[C::kMaxLevels], ncl2 = 0.f;
        // the first tile from f on (j: its index in its head) with level bits in the window
        auto next_tile = [&](int f, int& j) {
            int bh_ = 0;
            while (f < t1 && lbits(j) == 0) {
                f++;
                step(j, bh_);
            }
            return f;
        };
        // factors of tile fn (level bits nb) into nlam / ndt / ncl2
#define LLA_DNODE_FETCH(fn, nb)                                                   \
    do {                                                                          \
        const size_t r_ = static_cast<size_t>(fn) * kTile + row;                  \
        ncl2 = tok_cl2[r_];                                                       \
        _Pragma("unroll") for (int q = 0; q < C::kMaxLevels; q++) {               \
            const bool on_ = ((nb) >> q) & 1u;                                    \
            nlam[q] = on_ ? lambda[r_ * L + 8 + p_lo + q] : 0.f;                  \
            ndt[q] = on_ ? dtab[static_cast<size_t>(fn) * 16 + p_lo + q] : 0.f;   \
        }                                                                         \
    } while (0)
        int jf = j0;
        int f = next_tile(t0, jf);
        if (f < t1) LLA_DNODE_FETCH(f, lbits(jf));
        int rs = 0, ss = 0;
        uint32_t rph = 0, sph = 0;
        int n_sc = 0;
        while (f < t1) {
            if (__any_sync(0xffffffffu, *fail != 0)) break;
            const uint32_t bits = lbits(jf);
            cl2 = ncl2;
#pragma unroll
            for (int q = 0; q < C::kMaxLevels; q++) {
                lam[q] = nlam[q];
                dt[q] = ndt[q];
            }
            int jn = jf, bh_n = 0;
            step(jn, bh_n);
            const int fn = next_tile(f + 1, jn);
            if (fn < t1) LLA_DNODE_FETCH(fn, lbits(jn));
            if (!warp_wait(&raw_full[rs], rph)) {
                if (lane == 0) fail_now();
                break;
            }
#pragma unroll
            for (int q = 0; q < C::kMaxLevels; q++)
                if ((bits >> q) & 1u) w_sh[q][row] = lam[q] * exp2f(cl2 + dt[q]);
            const uint8_t* drow = smem + rs * C::kRawBytes + C::kQBytes + row * 128;
            uint4 x[8];
#pragma unroll
            for (int ch = 0; ch < 8; ch++) x[ch] = *reinterpret_cast<const uint4*>(drow + ((ch ^ (row & 7)) << 4));
            bool ok = true;
#pragma unroll 1
            for (uint32_t b = bits; b != 0; b &= b - 1) {
                const float w = w_sh[__ffs(b) - 1][row];
                if (n_sc >= C::kScaled && !warp_wait(&sc_empty[ss], sph ^ 1u)) {
                    ok = false;
                    break;
                }
                uint8_t* srow = scaled + ss * kPanelBytes + row * 128;
#pragma unroll
                for (int ch = 0; ch < 8; ch++) {
                    const float2 a0 = unpack_bf16(x[ch].x), a1 = unpack_bf16(x[ch].y), a2 = unpack_bf16(x[ch].z),
                                 a3 = unpack_bf16(x[ch].w);
                    *reinterpret_cast<uint4*>(srow + ((ch ^ (row & 7)) << 4)) =
                        make_uint4(pack_bf16(a0.x * w, a0.y * w), pack_bf16(a1.x * w, a1.y * w),
                                   pack_bf16(a2.x * w, a2.y * w), pack_bf16(a3.x * w, a3.y * w));
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sc_full[ss]);
                n_sc++;
                if (++ss == C::kScaled) {
                    ss = 0;
                    sph ^= 1u;
                }
            }
            if (!ok) {
                if (lane == 0) fail_now();
                break;
            }
            if (++rs == C::kRaw) {
                rs = 0;
                rph ^= 1u;
            }
            f = fn;
            jf = jn;
        }
#undef LLA_DNODE_FETCH
    } else if (warp >= 8) {
        const int quad = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        uint8_t* stage = drain_stage + quad * C::kDrainBytes;
        uint32_t par = 0, cut = 0;  // cut: the slot's current run began in another CTA
        int j = j0, bh = bh0;
        for (int f = t0; f < t1; f++, step(j, bh)) {
            const DnodeTile dt = dnode_tile(f, bh, j, NT, p_lo, np, t0, t1);
            cut = (cut & ~dt.start) | dt.start_cut;
            if (dt.end == 0) continue;
            if (__any_sync(0xffffffffu, *fail != 0)) break;
            bool ok = true;
#pragma unroll 1
            for (uint32_t b = dt.end; b != 0; b &= b - 1) {
                const int q = __ffs(b) - 1;
                if (!warp_wait(&acc_full[q], (par >> q) & 1u)) {
                    ok = false;
                    break;
                }
                par ^= 1u << q;
                tc_fence_after();
                float x[64];
                tmem_ld32(tmem + lane_base + q * kDV, x);
                tmem_ld32(tmem + lane_base + q * kDV + 32, x + 32);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&acc_empty[q]);
                    bulk_wait_read0();  // the previous reduce has read the staging box
                }
                __syncwarp();
                // row `lane` of this warp's 32: columns 32h + 4c .. + 3 at box h, chunk c ^ (lane & 7)
#pragma unroll
                for (int h = 0; h < 2; h++)
#pragma unroll
                    for (int c = 0; c < 8; c++)
                        *reinterpret_cast<float4*>(stage + h * 4096 + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                            make_float4(x[32 * h + 4 * c], x[32 * h + 4 * c + 1], x[32 * h + 4 * c + 2],
                                        x[32 * h + 4 * c + 3]);
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const int p = p_lo + q;
                    const int m = (dt.j >> p) - 1;
                    const int row0 = (dt.bh * node_count + lo_sh[p] + (m >> 1)) * kDk + quad * 32;
                    if (((cut | dt.end_cut) >> q) & 1u) {  // shared with a neighbour: add into the zeroed node
                        tma_reduce_add_2d(&tm_dn, stage, 0, row0);
                        tma_reduce_add_2d(&tm_dn, stage + 4096, 32, row0);
                    } else {  // the whole reading block: this CTA is the node's only writer
                        tma_store_2d(&tm_dn, stage, 0, row0);
                        tma_store_2d(&tm_dn, stage + 4096, 32, row0);
                    }
                    bulk_commit();
                }
            }
            if (!ok) {
                if (lane == 0) fail_now();
                break;
            }
        }
        if (lane == 0) bulk_wait0();
    }

    __syncthreads();
    if (*fail && warp == 0 && lane == 0) {
        for (int i = issued - C::kRaw > 0 ? issued - C::kRaw : 0; i < issued; i++)
            mbar_wait(&raw_full[i % C::kRaw], (i / C::kRaw) & 1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, tmem_cols);
}

// Zero the nodes whose reading block a CTA boundary of tc_dnode cuts (the only ones written by
// reduce-adds). grid (CTAs - 1, P), 256 threads: boundary b starts CTA b's share at tile f; for
// each set bit p of its tile index j with nonzero bits below p, the node (p, (j >> p) - 1) is cut.
__global__ void __launch_bounds__(256) tc_dnode_zero_cut_kernel(float* __restrict__ dnodes, int NT, int total,
                                                                int ctas, int node_count,
                                                                const __grid_constant__ Offsets lo) {
    const int b = blockIdx.x + 1, p = blockIdx.y;
    const int f = static_cast<int>(static_cast<int64_t>(b) * total / ctas);
    const int bh = f / NT, j = f - bh * NT;
    if (!((j >> p) & 1) || (j & ((1 << p) - 1)) == 0) return;
    float4* dst = reinterpret_cast<float4*>(
        dnodes + (static_cast<size_t>(bh) * node_count + lo.off[p] + (((j >> p) - 1) >> 1)) * kMsz);
    for (int i = threadIdx.x; i < kMsz / 4; i += blockDim.x) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ------------------------------------------------------------------ tc_cmat

// C_i = sum over the read ancestors (p, i >> p) of key tile i of
// exp(sum of the tile decays after i up to the node's last tile) dB_{p, i>>p},
// bf16 [BH][NT][dk][dv]. grid (NT, BH), 256 threads: warp w finds the weights of levels
// w, w + 8 (a warp-wide sum each), then every thread forms 32 elements (8 float4s).
__global__ void __launch_bounds__(256) tc_cmat_kernel(const float* __restrict__ dnodes, const float* __restrict__ g,
                                                      __nv_bfloat16* __restrict__ cmat, int NT, int P, int node_count,
                                                      const __grid_constant__ Offsets lo, int* __restrict__ item_counter) {
    __shared__ float wsh[32];
    __shared__ int rsh[32];
    const int i = blockIdx.x, bh = blockIdx.y;
    // the next kernel's item counter (this kernel runs before it on the same stream)
    if (i == 0 && bh == 0 && threadIdx.x == 0) *item_counter = 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int p = warp; p < P; p += 8) {
        const int m = i >> p;
        const bool read = (m & 1) == 0 && ((m + 1) << p) < NT;
        const int end = (m + 1) << p;  // one past the node's last tile
        float sacc = 0.f;
        if (read)
            for (int u = i + 1 + lane; u < end; u += 32) sacc += g[static_cast<size_t>(bh) * NT + u];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sacc += __shfl_xor_sync(0xffffffffu, sacc, off);
        if (lane == 0) {
            wsh[p] = read ? expf(sacc) : 0.f;
            rsh[p] = read ? 1 : 0;
        }
    }
    __syncthreads();
    // thread x accumulates the float4s x + 256 k, k < 8, of the node: eight independent loads
    // in flight per level
    constexpr int kVec = kMsz / 4 / 256;
    float4 acc[kVec];
#pragma unroll
    for (int k = 0; k < kVec; k++) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p = 0; p < P; p++) {
        if (!rsh[p]) continue;
        const float w = wsh[p];
        const float4* src = reinterpret_cast<const float4*>(
                                dnodes + (static_cast<size_t>(bh) * node_count + lo.off[p] + ((i >> p) >> 1)) * kMsz) +
                            threadIdx.x;
        float4 x[kVec];
#pragma unroll
        for (int k = 0; k < kVec; k++) x[k] = src[256 * k];
#pragma unroll
        for (int k = 0; k < kVec; k++) {
            acc[k].x = fmaf(w, x[k].x, acc[k].x);
            acc[k].y = fmaf(w, x[k].y, acc[k].y);
            acc[k].z = fmaf(w, x[k].z, acc[k].z);
            acc[k].w = fmaf(w, x[k].w, acc[k].w);
        }
    }
    uint2* dst = reinterpret_cast<uint2*>(cmat + (static_cast<size_t>(bh) * NT + i) * kMsz) + threadIdx.x;
#pragma unroll
    for (int k = 0; k < kVec; k++)
        dst[256 * k] = make_uint2(pack_bf16(acc[k].x, acc[k].y), pack_bf16(acc[k].z, acc[k].w));
}

// ------------------------------------------------------------------ tc_bwd_tile

struct TileCfg {
    static constexpr int kQ = 0;                     // Q tile  [t][d], 2 panels
    static constexpr int kK = 2 * kPanelBytes;       // K tile  [s][d], 2 panels
    static constexpr int kV = 4 * kPanelBytes;       // V tile  [s][e], 1 panel
    static constexpr int kDO = 5 * kPanelBytes;      // dO tile [t][e], 1 panel
    static constexpr int kA = 6 * kPanelBytes;       // A [t][s] bf16, 2 panels; then dQ out
    static constexpr int kG = 8 * kPanelBytes;       // G [t][s] bf16, 2 panels; then r_p o dO; then dK out
    static constexpr int kC = 10 * kPanelBytes;      // C_i [d][e] (copied with the inputs); then node slot 0
    static constexpr int kN = 11 * kPanelBytes;      // w o V [s][e]; then node slot 1 (B_p [d][e]); then dV out
    static constexpr int kR = kG + kPanelBytes;      // G's second panel; G's two hold a level pair's r_p o dO
    static constexpr int kBytes = 12 * kPanelBytes + 1024;
    static constexpr uint32_t kTxIn = 7 * kPanelBytes;
    // TMEM columns: S and dP until the A/G epilogue; dK and Z from the key side's MMAs, which
    // run beside it; then dQ over S, Y over dP, and dV
    static constexpr uint32_t kS = 0, kDP = 128;
    static constexpr uint32_t kDQ = 0, kY = 128, kDK = 256, kDVc = 384, kZ = 448;
    static constexpr uint32_t kTmemCols = 512;
};

// Persistent, one CTA per SM; 256 threads: thread (quad = warp % 4, lane) owns row
// t = 32 quad + lane (= TMEM lane), half = warp / 4 picks half of the columns. Thread 0
// issues the TMA copies and the MMAs between block-wide phases. A CTA takes its first
// (head, tile) item by its index and the rest from item_counter (zero at launch). Once an
// item's inputs are dead (its last MMA done and read back) the next item's inputs are
// copied in, behind this item's output staging, stores and dlambda rows.
__global__ void __launch_bounds__(256, 1)
    tc_bwd_tile_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_nodes, const __grid_constant__ CUtensorMap tm_cmat,
                       const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
                       const __grid_constant__ CUtensorMap tm_dv,
                       const float* __restrict__ lambda, const float* __restrict__ tok_cl2,
                       const float* __restrict__ dtab, float* __restrict__ dlambda, float* __restrict__ dcum, int T,
                       int NT, int L, int P, int node_count, const __grid_constant__ Offsets lo, int n_items,
                       int* __restrict__ item_counter, int* err) {
    using C = TileCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar_in, bar_s, bar_m1, bar_node[2], bar_lv, bar_k, bar_d;
    __shared__ uint32_t tmem_base_sh;
    __shared__ __align__(16) float cl2_sh[kTile];
    __shared__ __align__(16) float lam_sh[kTile * 32];  // the tile's lambda rows [t][L], L <= 32
    __shared__ float dlam8[kTile][8];
    __shared__ float dlamp[kTile][16];
    __shared__ float colE[kTile], dcs[kTile], zsh[kTile], wts[kTile];
    __shared__ __align__(16) float colw_sh[kTile];
    __shared__ float zpart[2][2][kTile];  // a level pair's q_t^T B_p dO_t, per round and column half
    __shared__ __align__(16) float dtab_sh[16];
    __shared__ int fail_sh, next_sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2;
    const int t = quad * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;

    if (tid == 0) {
        mbar_init(&bar_in, 1);
        mbar_init(&bar_s, 1);
        mbar_init(&bar_m1, 1);
        mbar_init(&bar_node[0], 1);
        mbar_init(&bar_node[1], 1);
        mbar_init(&bar_lv, 1);
        mbar_init(&bar_k, 1);
        mbar_init(&bar_d, 1);
        fence_mbar_init();
        fail_sh = 0;
    }
    if (warp == 0) tmem_alloc(&tmem_base_sh, C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    // every wait is warp-uniform and bounded; a failure is shared through fail_sh
    auto ok_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (warp_wait(bar, parity)) return true;
        if (lane == 0 && atomicExch(&fail_sh, 1) == 0) record_error(err, kDevTimeout);
        return false;
    };
    // row t of the 32 TMEM columns col + 32 half .. of this thread's lanes against the same
    // columns of V's row t (this half's share of the dot product)
    auto tmem_row_dot_v = [&](uint32_t col) -> float {
        float zv[32];
        tmem_ld32(tmem + lane_base + col + 32 * half, zv);
        const uint8_t* src = smem + C::kV;
        float y = 0.f;
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const uint4 x = *reinterpret_cast<const uint4*>(src + sw128_off(t, 4 * half + q));
            const float2 a0 = unpack_bf16(x.x), a1 = unpack_bf16(x.y), a2 = unpack_bf16(x.z), a3 = unpack_bf16(x.w);
            y = fmaf(zv[8 * q], a0.x, y); y = fmaf(zv[8 * q + 1], a0.y, y);
            y = fmaf(zv[8 * q + 2], a1.x, y); y = fmaf(zv[8 * q + 3], a1.y, y);
            y = fmaf(zv[8 * q + 4], a2.x, y); y = fmaf(zv[8 * q + 5], a2.y, y);
            y = fmaf(zv[8 * q + 6], a3.x, y); y = fmaf(zv[8 * q + 7], a3.y, y);
        }
        return y;
    };
    // thread 0: item it's inputs, C_i, and the per-row scalars: lambda rows (one contiguous
    // block of 128 L floats), the in-tile log2 decay prefix and the tile's level decay row
    auto issue_inputs = [&](int it) {
        const int ibh = it / NT, ij = it - ibh * NT;
        const int ir0 = ibh * T + ij * kTile;
        uint8_t* st = smem;
        mbar_expect_tx(&bar_in, C::kTxIn + kTile * L * 4 + kTile * 4 + 16 * 4);
        bulk_load(lam_sh, lambda + static_cast<size_t>(ir0) * L, kTile * L * 4, &bar_in);
        bulk_load(cl2_sh, tok_cl2 + ir0, kTile * 4, &bar_in);
        bulk_load(dtab_sh, dtab + (static_cast<size_t>(ibh) * NT + ij) * 16, 16 * 4, &bar_in);
        tma_load_2d(st + C::kQ, &tm_q, &bar_in, 0, ir0);
        tma_load_2d(st + C::kQ + kPanelBytes, &tm_q, &bar_in, 64, ir0);
        tma_load_2d(st + C::kK, &tm_k, &bar_in, 0, ir0);
        tma_load_2d(st + C::kK + kPanelBytes, &tm_k, &bar_in, 64, ir0);
        tma_load_2d(st + C::kV, &tm_v, &bar_in, 0, ir0);
        tma_load_2d(st + C::kDO, &tm_do, &bar_in, 0, ir0);
        tma_load_2d(st + C::kC, &tm_cmat, &bar_in, 0, (ibh * NT + ij) * kDk);
    };
    auto zero_sums = [&]() {
        for (int x = tid; x < kTile * 8; x += blockDim.x) (&dlam8[0][0])[x] = 0.f;
        for (int x = tid; x < kTile * 16; x += blockDim.x) (&dlamp[0][0])[x] = 0.f;
        if (tid < kTile) {
            colE[tid] = 0.f;
            dcs[tid] = 0.f;
            zsh[tid] = 0.f;
        }
    };

    // thread 0's copy bookkeeping, for the drain after a failed wait
    int in_issued = 0, in_waited = 0;
    int node_issued0 = 0, node_issued1 = 0, node_waited0 = 0, node_waited1 = 0;  // per node slot
    int claimed = 0;     // thread 0: the item claimed to follow this one
    bool k_bad = false;  // this thread saw a wait for the key side's MMAs run out
    int item = blockIdx.x;
    if (tid == 0 && item < n_items) {
        issue_inputs(item);
        in_issued = 1;
    }
    zero_sums();
    bool ok = true;
    uint32_t li = 0;  // level rounds so far: uses of bar_lv
    for (uint32_t ip = 0; item < n_items; ip++) {
    const int bh = item / NT, j = item - bh * NT;
    const int r0 = bh * T + j * kTile;
    const unsigned lvbits = static_cast<unsigned>(j) & ((1u << P) - 1u);
    const uint32_t par = ip & 1u;  // bar_in, bar_s, bar_m1, bar_k: one use per item
    auto node_row = [&](int p) { return (bh * node_count + lo.off[p] + (((j >> p) - 1) >> 1)) * kDk; };
    const int nrounds = __popc(lvbits);
    auto round_level = [&](int r) {  // the set bit of j that level round r reads
        unsigned b = lvbits;
        for (int k = 0; k < r; k++) b &= b - 1;
        return __ffs(b) - 1;
    };
    // thread 0: round r's node into slot r & 1 (C or N, adjacent panels, so a level pair's two
    // nodes form one 128-column operand; both are free once the key side's MMAs are done)
    auto issue_node = [&](int r) {
        const int sl = r & 1;
        mbar_expect_tx(&bar_node[sl], kPanelBytes);
        tma_load_2d(smem + (sl ? C::kN : C::kC), &tm_nodes, &bar_node[sl], 0, node_row(round_level(r)));
        if (sl) node_issued1++; else node_issued0++;
    };
    // the previous item's tensor stores have read A, G and N before this item writes there
    if (tid == 0) bulk_wait_read0();
    // ok stays block-uniform: every change goes through a barrier reduction
    ok = __syncthreads_and(ok && ok_wait(&bar_in, par));
    if (!ok) break;
    if (tid == 0) in_waited++;
    // decay from each key to the end of its 32-key block (the factorised decay of E1); read
    // after the barrier that follows the S and dP MMAs
    if (tid < kTile) colw_sh[tid] = exp2f(cl2_sh[tid | 31] - cl2_sh[tid]);
    // ---- S = Q K^T, dP = dO V^T
    if (tid == 0 && ok) {
        tc_fence_after();
        constexpr uint32_t kIdSS = idesc_bf16(kTile, kTile, 0, 0);
        const uint32_t qb = smem_u32(smem + C::kQ), kb = smem_u32(smem + C::kK);
        const uint32_t vb = smem_u32(smem + C::kV), ob = smem_u32(smem + C::kDO);
#pragma unroll
        for (int kk = 0; kk < kDk / 16; kk++) {
            const uint32_t off = (kk >> 2) * kPanelBytes + (kk & 3) * 32;
            mma_bf16(tmem + C::kS, sdesc(qb + off, 16, 1024), sdesc(kb + off, 16, 1024), kIdSS, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < kDV / 16; kk++) {
            mma_bf16(tmem + C::kDP, sdesc(ob + kk * 32, 16, 1024), sdesc(vb + kk * 32, 16, 1024), kIdSS,
                     kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar_s);
    }
    // ---- key side, beside S and dP: dK = (w o V) C_i^T and Z = K C_i (C_i came with the
    // inputs); the key side's dV term (w o K) C_i is diag(w) Z, added when dV is staged.
    // w o V (row t = key s, this half's 32 columns) goes to N while S and dP run.
    {
        const float w = exp2f(cl2_sh[kTile - 1] - cl2_sh[t]);
        if (half == 0) wts[t] = w;
        const uint8_t* src = smem + C::kV;
        uint8_t* dst = smem + C::kN;
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const uint32_t off = sw128_off(t, 4 * half + q);
            const uint4 x = *reinterpret_cast<const uint4*>(src + off);
            const float2 a0 = unpack_bf16(x.x), a1 = unpack_bf16(x.y), a2 = unpack_bf16(x.z), a3 = unpack_bf16(x.w);
            *reinterpret_cast<uint4*>(dst + off) =
                make_uint4(pack_bf16(a0.x * w, a0.y * w), pack_bf16(a1.x * w, a1.y * w),
                           pack_bf16(a2.x * w, a2.y * w), pack_bf16(a3.x * w, a3.y * w));
        }
    }
    fence_async_smem();
    ok = __syncthreads_and(ok && ok_wait(&bar_s, par));
    tc_fence_after();
    // thread 0 (lane quadrant 0, the lightest share of the epilogue below) issues the key
    // side's MMAs; they run beside the epilogue
    if (tid == 0 && ok) {
        const uint32_t rb = smem_u32(smem + C::kN), cb = smem_u32(smem + C::kC);
        const uint32_t kb = smem_u32(smem + C::kK);
        constexpr uint32_t kIdK = idesc_bf16(kTile, kDk, 0, 0);
        constexpr uint32_t kIdV = idesc_bf16(kTile, kDV, 0, 1);
#pragma unroll
        for (int kk = 0; kk < kDV / 16; kk++)
            mma_bf16(tmem + C::kDK, sdesc(rb + kk * 32, 16, 1024), sdesc(cb + kk * 32, 16, 1024), kIdK,
                     kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kDk / 16; kk++) {
            const uint32_t off = (kk >> 2) * kPanelBytes + (kk & 3) * 32;
            mma_bf16(tmem + C::kZ, sdesc(kb + off, 16, 1024), sdesc(cb + kk * 2048, kPanelBytes, 1024), kIdV,
                     kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar_k);
        // the item to follow
        claimed = static_cast<int>(gridDim.x) + atomicAdd(item_counter, 1);
    }

    // ---- E1: A, G (bf16), dlambda levels 0..7, the decay derivatives' row sums. The two
    // warps of a lane quadrant take alternate 16-key halves of every 32-key block, so the
    // masked diagonal block of the quadrant is shared evenly between them. The decay
    // derivative of pair (t, s) is E = A (o) dP: its row sums (here) and column sums (from
    // dV's accumulator, below) both take A as rounded to bf16 for the MMAs, so that the pairs
    // the suffix sums of dlog_a cancel cancel exactly.
    // row t's sum over this half's 16 keys of A[t][s] dP[t][s], A as packed in pa
    auto rowsum_a = [&](const uint32_t (&pa)[8], const float (&dpv)[16]) {
        float r = 0.f;
#pragma unroll
        for (int e = 0; e < 8; e++) {
            const float2 a = unpack_bf16(pa[e]);
            r = fmaf(a.x, dpv[2 * e], r);
            r = fmaf(a.y, dpv[2 * e + 1], r);
        }
        return r;
    };
    if (ok) {
        const float cl2_t = cl2_sh[t];
        float dl[8];
#pragma unroll
        for (int l = 0; l < 8; l++) dl[l] = 0.f;
        float rowE = 0.f;
#pragma unroll 1
        for (int c = 0; c < 4; c++) {
            const int cb32 = 32 * c;             // the 32-key block
            const int cb = cb32 + 16 * half;     // this warp's 16 keys of it
            uint32_t pa[8], pg[8];
            const bool zero = cb32 > quad * 32;  // every key after every row of this warp
            if (zero) {
#pragma unroll
                for (int e = 0; e < 8; e++) pa[e] = pg[e] = 0u;
            } else if (cb32 < quad * 32) {
                // every key of the block precedes every row of this warp: one level per row
                // (t and s differ first in bit 5 or 6) and decay exp2(cl_t - cl_end) colw[s]
                float sv[16], dpv[16];
                tmem_ld16(tmem + lane_base + C::kS + cb, sv);
                tmem_ld16(tmem + lane_base + C::kDP + cb, dpv);
                const int l = 32 - __clz(t ^ cb32);
                float lm = lam_sh[t * L];
#pragma unroll
                for (int ll = 1; ll < 8; ll++) lm = (l == ll) ? lam_sh[t * L + ll] : lm;
                const float rowf = exp2f(cl2_t - cl2_sh[cb32 + 31]);
                float dsum = 0.f;
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    const float D0 = rowf * colw_sh[cb + e], D1 = rowf * colw_sh[cb + e + 1];
                    const float s0 = D0 * sv[e], s1 = D1 * sv[e + 1];
                    const float q0 = s0 * dpv[e], q1 = s1 * dpv[e + 1];
                    dsum += q0 + q1;
                    pa[e >> 1] = pack_bf16(lm * s0, lm * s1);
                    pg[e >> 1] = pack_bf16(lm * D0 * dpv[e], lm * D1 * dpv[e + 1]);
                }
                rowE += rowsum_a(pa, dpv);
#pragma unroll
                for (int ll = 0; ll < 8; ll++) dl[ll] += (l == ll) ? dsum : 0.f;
            } else if (cl2_sh[cb32] - cl2_sh[cb32 + 31] < 100.f) {
                // the diagonal 32-key block (t and s share bits 5 and 6, so the levels are 0..5)
                // with the block's decay under 2^100: decay exp2(cl_t - cl_end) colw[s], both
                // factors within 2^(+-100). With m = t mod 16, a lane whose 16-key group is
                // this half's sees level bitlength(m ^ k) at key k and keeps keys k <= m; a
                // lane of the other group sees level 5 everywhere and keeps every key (half 0)
                // or none (half 1).
                float sv[16], dpv[16];
                tmem_ld16(tmem + lane_base + C::kS + cb, sv);
                tmem_ld16(tmem + lane_base + C::kDP + cb, dpv);
                const int m = lane & 15;
                const bool same = ((lane >> 4) & 1) == half;
                const int klim = same ? m : (half == 0 ? 15 : -1);
                float w[6];
#pragma unroll
                for (int ll = 0; ll < 6; ll++) w[ll] = lam_sh[t * L + ll];
#pragma unroll
                for (int ll = 0; ll < 5; ll++) w[ll] = same ? w[ll] : w[5];
                // lambda at each key by the bits of m ^ k, lowest bit first
                const bool m0 = m & 1, m1 = (m >> 1) & 1, m2 = (m >> 2) & 1, m3 = (m >> 3) & 1;
                float w1x[2], w2x[4], w3x[8], lmk[16];
#pragma unroll
                for (int b = 0; b < 2; b++) w1x[b] = (b != static_cast<int>(m0)) ? w[1] : w[0];
#pragma unroll
                for (int b = 0; b < 4; b++) w2x[b] = ((b >> 1) != static_cast<int>(m1)) ? w[2] : w1x[b & 1];
#pragma unroll
                for (int b = 0; b < 8; b++) w3x[b] = ((b >> 2) != static_cast<int>(m2)) ? w[3] : w2x[b & 3];
#pragma unroll
                for (int b = 0; b < 16; b++) lmk[b] = ((b >> 3) != static_cast<int>(m3)) ? w[4] : w3x[b & 7];
                const float rowf = exp2f(cl2_t - cl2_sh[cb32 + 31]);
                float cw[16];
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const float4 c4 = *reinterpret_cast<const float4*>(colw_sh + cb + 4 * q);
                    cw[4 * q] = c4.x;
                    cw[4 * q + 1] = c4.y;
                    cw[4 * q + 2] = c4.z;
                    cw[4 * q + 3] = c4.w;
                }
                float x[16];  // D S dP per key
#pragma unroll
                for (int k = 0; k < 16; k += 2) {
                    float av[2], gv[2];
#pragma unroll
                    for (int h = 0; h < 2; h++) {
                        const float D = k + h <= klim ? rowf * cw[k + h] : 0.f;
                        const float ds = D * sv[k + h];
                        x[k + h] = ds * dpv[k + h];
                        av[h] = lmk[k + h] * ds;
                        gv[h] = lmk[k + h] * D * dpv[k + h];
                    }
                    pa[k >> 1] = pack_bf16(av[0], av[1]);
                    pg[k >> 1] = pack_bf16(gv[0], gv[1]);
                }
                // per-level sums: level l > 0 of the own group is the 2^(l-1) keys whose bits
                // above l - 1 match m's and whose bit l - 1 does not
                float g2[8], g4[4], g8[2];
#pragma unroll
                for (int b = 0; b < 8; b++) g2[b] = x[2 * b] + x[2 * b + 1];
#pragma unroll
                for (int b = 0; b < 4; b++) g4[b] = g2[2 * b] + g2[2 * b + 1];
#pragma unroll
                for (int b = 0; b < 2; b++) g8[b] = g4[2 * b] + g4[2 * b + 1];
                const float tot = g8[0] + g8[1];
                float y0[8], y1[8];  // pairs picked by bit 0: the key m's side, the other side
#pragma unroll
                for (int b = 0; b < 8; b++) {
                    y0[b] = m0 ? x[2 * b + 1] : x[2 * b];
                    y1[b] = m0 ? x[2 * b] : x[2 * b + 1];
                }
                auto pick8 = [&](const float (&v)[8], bool b0, bool b1, bool b2) {
                    const float a0 = b0 ? v[1] : v[0], a1 = b0 ? v[3] : v[2];
                    const float a2 = b0 ? v[5] : v[4], a3 = b0 ? v[7] : v[6];
                    const float c0 = b1 ? a1 : a0, c1 = b1 ? a3 : a2;
                    return b2 ? c1 : c0;
                };
                const float l0 = pick8(y0, m1, m2, m3);   // key m
                const float l1 = pick8(y1, m1, m2, m3);   // key m ^ 1
                const float l2 = pick8(g2, !m1, m2, m3);  // keys m ^ 2, m ^ 3
                const float l3 = m2 ? (m3 ? g4[2] : g4[0]) : (m3 ? g4[3] : g4[1]);
                const float l4 = m3 ? g8[0] : g8[1];
                dl[0] += same ? l0 : 0.f;
                dl[1] += same ? l1 : 0.f;
                dl[2] += same ? l2 : 0.f;
                dl[3] += same ? l3 : 0.f;
                dl[4] += same ? l4 : 0.f;
                dl[5] += same ? 0.f : tot;
                rowE += rowsum_a(pa, dpv);
            } else {
                // the diagonal 32-key block with a decay over 2^100 across it: one exp2 per key
                float sv[16], dpv[16];
                tmem_ld16(tmem + lane_base + C::kS + cb, sv);
                tmem_ld16(tmem + lane_base + C::kDP + cb, dpv);
                float lr[6];
#pragma unroll
                for (int ll = 0; ll < 6; ll++) lr[ll] = lam_sh[t * L + ll];
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    float av[2], gv[2];
#pragma unroll
                    for (int h = 0; h < 2; h++) {
                        const int s = cb + e + h;
                        const int l = 32 - __clz(t ^ s);
                        float lm = lr[0];
#pragma unroll
                        for (int ll = 1; ll < 6; ll++) lm = (l == ll) ? lr[ll] : lm;
                        // decay, zero for keys after t (masked)
                        const float D = s <= t ? exp2f(fminf(cl2_t - cl2_sh[s], 0.f)) : 0.f;
                        const float ds = D * sv[e + h];
                        const float dq_ = ds * dpv[e + h];
#pragma unroll
                        for (int ll = 0; ll < 6; ll++) dl[ll] += (l == ll) ? dq_ : 0.f;
                        av[h] = lm * ds;
                        gv[h] = lm * D * dpv[e + h];
                    }
                    pa[e >> 1] = pack_bf16(av[0], av[1]);
                    pg[e >> 1] = pack_bf16(gv[0], gv[1]);
                }
                rowE += rowsum_a(pa, dpv);
            }
            uint8_t* pA = smem + C::kA + (cb >> 6) * kPanelBytes;
            uint8_t* pG = smem + C::kG + (cb >> 6) * kPanelBytes;
            const int ch0 = (cb & 63) >> 3;
#pragma unroll
            for (int q = 0; q < 2; q++) {
                *reinterpret_cast<uint4*>(pA + sw128_off(t, ch0 + q)) =
                    make_uint4(pa[4 * q], pa[4 * q + 1], pa[4 * q + 2], pa[4 * q + 3]);
                *reinterpret_cast<uint4*>(pG + sw128_off(t, ch0 + q)) =
                    make_uint4(pg[4 * q], pg[4 * q + 1], pg[4 * q + 2], pg[4 * q + 3]);
            }
        }
#pragma unroll
        for (int l = 0; l < 8; l++)
            if (dl[l] != 0.f) atomicAdd(&dlam8[t][l], dl[l]);
        atomicAdd(&dcs[t], rowE);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- dV = A^T dO, dQ = G K, dK += G^T Q (onto the key side's term)
    if (tid == 0 && ok) {
        tc_fence_after();
        const uint32_t ab = smem_u32(smem + C::kA), gb = smem_u32(smem + C::kG);
        const uint32_t qb = smem_u32(smem + C::kQ), kb = smem_u32(smem + C::kK), ob = smem_u32(smem + C::kDO);
        constexpr uint32_t kIdV = idesc_bf16(kTile, kDV, 1, 1);
        constexpr uint32_t kIdQ = idesc_bf16(kTile, kDk, 0, 1);
        constexpr uint32_t kIdK = idesc_bf16(kTile, kDk, 1, 1);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; kk++) {
            const uint32_t koff = (kk >> 2) * kPanelBytes + (kk & 3) * 32;
            mma_bf16(tmem + C::kDVc, sdesc(ab + kk * 2048, kPanelBytes, 1024), sdesc(ob + kk * 2048, kPanelBytes, 1024),
                     kIdV, kk > 0 ? 1u : 0u);
            mma_bf16(tmem + C::kDQ, sdesc(gb + koff, 16, 1024), sdesc(kb + kk * 2048, kPanelBytes, 1024), kIdQ,
                     kk > 0 ? 1u : 0u);
            mma_bf16(tmem + C::kDK, sdesc(gb + kk * 2048, kPanelBytes, 1024), sdesc(qb + kk * 2048, kPanelBytes, 1024),
                     kIdK, 1u);
        }
        mma_commit(&bar_m1);
        // N and C are free once the key side's MMAs are done: the first two rounds' nodes
        if (mbar_wait(&bar_k, par)) {
            if (nrounds > 0) issue_node(0);
            if (nrounds > 1) issue_node(1);
        } else {
            k_bad = true;
            if (atomicExch(&fail_sh, 1) == 0) record_error(err, kDevTimeout);
        }
    }

    // Z's row sums with V (for dcum) while the MMAs above run
    if (ok && ok_wait(&bar_k, par)) {
        tc_fence_after();
        atomicAdd(&zsh[t], tmem_row_dot_v(C::kZ));
    } else {
        k_bad = true;
    }
    tc_fence_before();
    ok = __syncthreads_and(ok && ok_wait(&bar_m1, par) && !k_bad);
    tc_fence_after();
    // the column sums of E: for key s, sum_t A[t][s] (dO_t . V_s) = (A^T dO)[s,:] . V_s, dV's
    // accumulator (before the key side's term, added when dV is staged) against V
    if (ok) atomicAdd(&colE[t], tmem_row_dot_v(C::kDVc));
    // ---- query side: one round per set bit p of j, lowest first, in pairs. Rounds 2k and
    // 2k + 1 read their nodes from slots C and N and their r o dO from G's two panels: one
    // N = 128 chain gives both Y_p = Q B_p, one K = 128 chain adds both (r_p o dO) B_p^T to
    // dQ. The first pair's copies went out with the MMAs above, the next pair's go out when a
    // pair is done; its r o dO is scaled while this pair's Y is read back, and the row sums go
    // through zpart: one block barrier per pair.
    {
        const float cl2_t = cl2_sh[t];
        // r o dO, row t, this half's 32 columns (chunks 4 half .. 4 half + 3), into panel dst
        auto scale_rdo = [&](int dst_off, float rr) {
            const uint8_t* src = smem + C::kDO;
            uint8_t* dst = smem + dst_off;
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const uint32_t off = sw128_off(t, 4 * half + q);
                const uint4 x = *reinterpret_cast<const uint4*>(src + off);
                const float2 a0 = unpack_bf16(x.x), a1 = unpack_bf16(x.y), a2 = unpack_bf16(x.z), a3 = unpack_bf16(x.w);
                *reinterpret_cast<uint4*>(dst + off) =
                    make_uint4(pack_bf16(a0.x * rr, a0.y * rr), pack_bf16(a1.x * rr, a1.y * rr),
                               pack_bf16(a2.x * rr, a2.y * rr), pack_bf16(a3.x * rr, a3.y * rr));
            }
        };
        // round r's level, its decay rho and weight rr = lambda_t^(8+p) rho for row t
        auto weights = [&](int r, int& pp, float& rho_, float& rr_) {
            pp = round_level(r);
            rho_ = exp2f(cl2_t + dtab_sh[pp]);
            rr_ = lam_sh[t * L + 8 + pp] * rho_;
        };
        // this half's share of Y[t, col ..] . dO_t (32 columns)
        auto y_dot_do = [&](const uint32_t (&y0)[16], const uint32_t (&y1)[16]) {
            const uint8_t* src = smem + C::kDO;
            float z = 0.f;
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const uint32_t* yv = q < 2 ? y0 + 8 * q : y1 + 8 * (q - 2);
                const uint4 x = *reinterpret_cast<const uint4*>(src + sw128_off(t, 4 * half + q));
                const float2 a0 = unpack_bf16(x.x), a1 = unpack_bf16(x.y), a2 = unpack_bf16(x.z),
                             a3 = unpack_bf16(x.w);
                z = fmaf(__uint_as_float(yv[0]), a0.x, z); z = fmaf(__uint_as_float(yv[1]), a0.y, z);
                z = fmaf(__uint_as_float(yv[2]), a1.x, z); z = fmaf(__uint_as_float(yv[3]), a1.y, z);
                z = fmaf(__uint_as_float(yv[4]), a2.x, z); z = fmaf(__uint_as_float(yv[5]), a2.y, z);
                z = fmaf(__uint_as_float(yv[6]), a3.x, z); z = fmaf(__uint_as_float(yv[7]), a3.y, z);
            }
            return z;
        };
        float rho_a = 0.f, rr_a = 0.f, rho_b = 0.f, rr_b = 0.f;
        int p_a = 0, p_b = 0;
        if (nrounds > 0 && ok) {
            weights(0, p_a, rho_a, rr_a);
            scale_rdo(C::kG, rr_a);
            if (nrounds > 1) {
                weights(1, p_b, rho_b, rr_b);
                scale_rdo(C::kR, rr_b);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        for (int r = 0; r < nrounds && ok; r += 2) {
            const bool two = r + 1 < nrounds;
            if (tid == 0) {
                tc_fence_after();
                bool got = mbar_wait(&bar_node[0], node_waited0 & 1);
                if (got) node_waited0++;
                if (got && two) {
                    got = mbar_wait(&bar_node[1], node_waited1 & 1);
                    if (got) node_waited1++;
                }
                if (got) {
                    tc_fence_after();
                    const uint32_t qb = smem_u32(smem + C::kQ), gb = smem_u32(smem + C::kG);
                    const uint32_t cb = smem_u32(smem + C::kC);
                    const uint32_t idy = two ? idesc_bf16(kTile, 2 * kDV, 0, 1) : idesc_bf16(kTile, kDV, 0, 1);
                    constexpr uint32_t kIdX = idesc_bf16(kTile, kDk, 0, 0);
#pragma unroll
                    for (int kk = 0; kk < kDk / 16; kk++) {
                        const uint32_t off = (kk >> 2) * kPanelBytes + (kk & 3) * 32;
                        mma_bf16(tmem + C::kY, sdesc(qb + off, 16, 1024), sdesc(cb + kk * 2048, kPanelBytes, 1024),
                                 idy, kk > 0 ? 1u : 0u);
                    }
                    // K = 64 per round: rows of r o dO (panel G or R) against the node's rows (C or N)
                    const int nk = two ? 2 * kDV / 16 : kDV / 16;
#pragma unroll
                    for (int kk = 0; kk < 2 * kDV / 16; kk++) {
                        if (kk < nk) {
                            const uint32_t off = (kk >> 2) * kPanelBytes + (kk & 3) * 32;
                            mma_bf16(tmem + C::kDQ, sdesc(gb + off, 16, 1024), sdesc(cb + off, 16, 1024), kIdX, 1u);
                        }
                    }
                    mma_commit(&bar_lv);
                } else if (atomicExch(&fail_sh, 1) == 0) {
                    record_error(err, kDevTimeout);
                }
            }
            ok = __syncthreads_and(ok_wait(&bar_lv, li & 1));
            tc_fence_after();
            float rho_na = 0.f, rr_na = 0.f, rho_nb = 0.f, rr_nb = 0.f;
            int p_na = 0, p_nb = 0;
            if (ok) {
                if (tid == 0) {
                    if (r + 2 < nrounds) issue_node(r + 2);
                    if (r + 3 < nrounds) issue_node(r + 3);
                }
                uint32_t ya0[16], ya1[16], yb0[16], yb1[16];
                tmem_ld16_issue(tmem + lane_base + C::kY + 32 * half, ya0);
                tmem_ld16_issue(tmem + lane_base + C::kY + 32 * half + 16, ya1);
                if (two) {
                    tmem_ld16_issue(tmem + lane_base + C::kY + kDV + 32 * half, yb0);
                    tmem_ld16_issue(tmem + lane_base + C::kY + kDV + 32 * half + 16, yb1);
                }
                if (r + 2 < nrounds) {
                    weights(r + 2, p_na, rho_na, rr_na);
                    scale_rdo(C::kG, rr_na);
                    if (r + 3 < nrounds) {
                        weights(r + 3, p_nb, rho_nb, rr_nb);
                        scale_rdo(C::kR, rr_nb);
                    }
                }
                tmem_ld16_wait(ya0);
                tmem_ld16_wait(ya1);
                zpart[0][half][t] = y_dot_do(ya0, ya1);
                if (two) {
                    tmem_ld16_wait(yb0);
                    tmem_ld16_wait(yb1);
                    zpart[1][half][t] = y_dot_do(yb0, yb1);
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            if (ok && half == 0) {
                const float za = zpart[0][0][t] + zpart[0][1][t];
                dlamp[t][p_a] = rho_a * za;
                float d = rr_a * za;
                if (two) {
                    const float zb = zpart[1][0][t] + zpart[1][1][t];
                    dlamp[t][p_b] = rho_b * zb;
                    d += rr_b * zb;
                }
                dcs[t] += d;
            }
            rho_a = rho_na;
            rr_a = rr_na;
            p_a = p_na;
            rho_b = rho_nb;
            rr_b = rr_nb;
            p_b = p_nb;
            li++;
        }
    }

    // this item's inputs are dead (the last block barrier above follows their last reads and
    // MMAs): copy in the next item's
    if (tid == 0) {
        int next = n_items;
        if (ok) {
            next = claimed;
            if (next < n_items) {
                issue_inputs(next);
                in_issued++;
            }
        }
        next_sh = next;
    }

    // ---- outputs: dQ, dK, dV (bf16) into the now free A, G and N areas in the TMA layout,
    // then written by tensor stores; the decay derivative per row
    if (ok) {
        const size_t row = static_cast<size_t>(r0) + t;
        float x[32];
        auto put = [&](uint8_t* panel, int ch0) {
#pragma unroll
            for (int q = 0; q < 4; q++)
                *reinterpret_cast<uint4*>(panel + sw128_off(t, ch0 + q)) =
                    make_uint4(pack_bf16(x[8 * q], x[8 * q + 1]), pack_bf16(x[8 * q + 2], x[8 * q + 3]),
                               pack_bf16(x[8 * q + 4], x[8 * q + 5]), pack_bf16(x[8 * q + 6], x[8 * q + 7]));
        };
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
            tmem_ld32(tmem + lane_base + C::kDQ + 64 * half + c0, x);
            put(smem + C::kA + half * kPanelBytes, c0 >> 3);
            tmem_ld32(tmem + lane_base + C::kDK + 64 * half + c0, x);
            put(smem + C::kG + half * kPanelBytes, c0 >> 3);
        }
        // dV: A^T dO + diag(w) Z, w the key's decay to the tile end
        tmem_ld32(tmem + lane_base + C::kDVc + 32 * half, x);
        {
            float zv[32];
            tmem_ld32(tmem + lane_base + C::kZ + 32 * half, zv);
            const float w = wts[t];
#pragma unroll
            for (int i = 0; i < 32; i++) x[i] = fmaf(w, zv[i], x[i]);
        }
        put(smem + C::kN, 4 * half);
        if (half == 0) dcum[row] = dcs[t] - colE[t] - wts[t] * zsh[t];
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && ok) {
        tma_store_2d(&tm_dq, smem + C::kA, 0, r0);
        tma_store_2d(&tm_dq, smem + C::kA + kPanelBytes, 64, r0);
        tma_store_2d(&tm_dk, smem + C::kG, 0, r0);
        tma_store_2d(&tm_dk, smem + C::kG + kPanelBytes, 64, r0);
        tma_store_2d(&tm_dv, smem + C::kN, 0, r0);
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
    if (ok)
        for (int x = tid; x < kTile * L; x += blockDim.x) {
            const int row = x / L, l = x - row * L;
            dlambda[static_cast<size_t>(r0) * L + x] = l < 8 ? dlam8[row][l] : (l < 24 ? dlamp[row][l - 8] : 0.f);
        }
    __syncthreads();
    item = next_sh;
    zero_sums();
    if (!ok) break;
    }

    if (tid == 0) {
        // the tensor stores have read their shared-memory sources before it goes away
        bulk_wait_read0();
    }
    __syncthreads();
    if (tid == 0 && fail_sh) {
        // let this CTA's copies land before its shared memory goes away
        if (in_issued > in_waited) mbar_wait(&bar_in, (in_issued - 1) & 1);
        if (node_issued0 > node_waited0) mbar_wait(&bar_node[0], (node_issued0 - 1) & 1);
        if (node_issued1 > node_waited1) mbar_wait(&bar_node[1], (node_issued1 - 1) & 1);
    }
    if (tid == 0) {
        // every MMA issued above has completed before TMEM is released
        mma_commit(&bar_d);
        mbar_wait(&bar_d, 0);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, C::kTmemCols);
}

}  // namespace

bool tc_bwd_supported(int dtype, int dk, int dv, int T) {
    return dtype == 0 && dk == kDk && dv == kDV && T % kTile == 0;
}

size_t tc_bwd_workspace_bytes(const TcPlan& pl) {
    const size_t BH = static_cast<size_t>(pl.B) * pl.H;
    const size_t dnodes = (BH * pl.node_count * kMsz * sizeof(float) + 1023) / 1024 * 1024;
    const size_t cmat = (BH * pl.NT * kMsz * 2 + 1023) / 1024 * 1024;
    const size_t dcum = (BH * pl.T * sizeof(float) + 255) / 256 * 256;
    return pl.total_bytes + dnodes + cmat + dcum;
}

cudaError_t tc_backward(const TcPlan& pl, const void* q, const void* k, const void* v, const float* log_a,
                        const float* lambda, const void* dout, void* dq, void* dk, void* dv, float* dlog_a,
                        float* dlambda, void* workspace, int* err, cudaStream_t stream) {
    const int BH = pl.B * pl.H;
    const int L = bitlength(static_cast<int64_t>(pl.T) - 1) + 1;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const float* g_tiles = reinterpret_cast<const float*>(ws);
    const __nv_bfloat16* nodes = reinterpret_cast<const __nv_bfloat16*>(ws + pl.g_bytes);
    const float* dtab = reinterpret_cast<const float*>(ws + pl.g_bytes + pl.nodes_bytes + pl.seg_bytes);
    const float* tok_cl2 =
        reinterpret_cast<const float*>(ws + pl.g_bytes + pl.nodes_bytes + pl.seg_bytes + pl.dtab_bytes);
    const size_t dnodes_bytes = (static_cast<size_t>(BH) * pl.node_count * kMsz * sizeof(float) + 1023) / 1024 * 1024;
    const size_t cmat_bytes = (static_cast<size_t>(BH) * pl.NT * kMsz * 2 + 1023) / 1024 * 1024;
    float* dnodes = reinterpret_cast<float*>(ws + pl.total_bytes);
    __nv_bfloat16* cmat = reinterpret_cast<__nv_bfloat16*>(ws + pl.total_bytes + dnodes_bytes);
    float* dcum = reinterpret_cast<float*>(ws + pl.total_bytes + dnodes_bytes + cmat_bytes);
    Offsets lo;
    for (int p = 0; p < 32; p++) lo.off[p] = pl.level_off[p];

    cudaError_t e = tc_nodes_only(pl, k, v, log_a, workspace, err, stream);
    if (e != cudaSuccess) return e;

    const uint64_t rows = static_cast<uint64_t>(BH) * pl.T;
    CUtensorMap tq, tk, tv, tdo, tn, tc;
    if (!make_map(&tq, q, rows, kDk) || !make_map(&tk, k, rows, kDk) || !make_map(&tv, v, rows, kDV) ||
        !make_map(&tdo, dout, rows, kDV) ||
        !make_map(&tc, cmat, static_cast<uint64_t>(BH) * pl.NT * kDk, kDV))
        return cudaErrorInvalidValue;
    if (pl.node_count > 0) {
        if (!make_map(&tn, nodes, static_cast<uint64_t>(BH) * pl.node_count * kDk, kDV)) return cudaErrorInvalidValue;
    } else {
        tn = tc;  // never read: no tile has an earlier block
    }

    if (pl.node_count > 0) {
        CUtensorMap tdn;
        if (!make_map_f32_32x32(&tdn, dnodes, static_cast<uint64_t>(BH) * pl.node_count * kDk, kDV))
            return cudaErrorInvalidValue;
        const int total = BH * pl.NT;
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
            cudaGetLastError();
            sms = 152;
        }
        const int grid = total < sms ? total : sms;
        if (grid > 1) {
            tc_dnode_zero_cut_kernel<<<dim3(grid - 1, pl.P), 256, 0, stream>>>(dnodes, pl.NT, total, grid,
                                                                                pl.node_count, lo);
            note_launch(stream, "tc_dnode_zero_cut");
        }
        e = cudaFuncSetAttribute(tc_dnode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, DnodeCfg::kBytes);
        if (e != cudaSuccess) return e;
        // levels in windows of at most eight (one TMEM accumulator of 64 columns each)
        for (int p_lo = 0; p_lo < pl.P; p_lo += DnodeCfg::kMaxLevels) {
            const int np = pl.P - p_lo < DnodeCfg::kMaxLevels ? pl.P - p_lo : DnodeCfg::kMaxLevels;
            tc_dnode_kernel<<<grid, DnodeCfg::kThreads, DnodeCfg::kBytes, stream>>>(
                tq, tdo, tdn, lambda, tok_cl2, dtab, pl.T, pl.NT, L, pl.node_count, lo, p_lo, np, total, err);
            note_launch(stream, "tc_dnode");
        }
    }
    int* item_counter = reinterpret_cast<int*>(ws + pl.total_bytes - pl.ctr_bytes);
    tc_cmat_kernel<<<dim3(pl.NT, BH), 256, 0, stream>>>(dnodes, g_tiles, cmat, pl.NT, pl.P, pl.node_count, lo,
                                                         item_counter);
    note_launch(stream, "tc_cmat");
    e = cudaFuncSetAttribute(tc_bwd_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TileCfg::kBytes);
    if (e != cudaSuccess) return e;
    CUtensorMap tdq, tdk, tdv;
    if (!make_map(&tdq, dq, rows, kDk) || !make_map(&tdk, dk, rows, kDk) || !make_map(&tdv, dv, rows, kDV))
        return cudaErrorInvalidValue;
    const int n_items = BH * pl.NT;
    int tdev = 0, tsms = 0;
    if (cudaGetDevice(&tdev) != cudaSuccess ||
        cudaDeviceGetAttribute(&tsms, cudaDevAttrMultiProcessorCount, tdev) != cudaSuccess || tsms <= 0) {
        cudaGetLastError();
        tsms = 152;
    }
    const int tile_grid = n_items < tsms ? n_items : tsms;
    tc_bwd_tile_kernel<<<tile_grid, 256, TileCfg::kBytes, stream>>>(tq, tk, tv, tdo, tn, tc, tdq, tdk, tdv, lambda,
                                                                    tok_cl2, dtab, dlambda, dcum, pl.T, pl.NT, L, pl.P,
                                                                    pl.node_count, lo, n_items, item_counter, err);
    note_launch(stream, "tc_bwd_tile");
    return bwd_dloga(dcum, dlog_a, BH, pl.T, stream);
}

}  // namespace lla
