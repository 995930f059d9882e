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
//   * the keys of tile Pt (tokens 128 Pt .. pos) have levels 0..7: that tile
//     is visited once per level held at pos (at most 8 "virtual" tiles), each
//     time with the weights of the other levels (and of tokens past pos) zero.
// Kernels (one stream, in order):
//   state_tile_totals : g_u = sum of log_a over full tile u.
//   state_offsets     : each sequence's first item in the flattened tile list
//                       (sequences may have different lengths: packed input).
//   state_prep        : per head, tail_u = sum of log_a from the end of tile u
//                       to pos (reverse scan, newest first). The held slots need
//                       no zeroing: each has at least one tile and is written
//                       exactly once (by tc_state or state_fixup).
//   tc_state          : persistent; each CTA takes an equal share of the
//                       flattened (head, tile) list. Per tile,
//                       w_s = exp(tail_u + decay from s to the tile end), and
//                       w o V is split into bf16 hi + lo (so the product keeps
//                       ~16 mantissa bits); one tcgen05 MMA per 16-token step
//                       (N = 2 dv: both parts side by side) accumulates
//                       K^T [hi | lo] in TMEM, and the two halves are summed
//                       when the accumulator is drained. A run of tiles of one
//                       slot that lies within one CTA's share is stored into the
//                       slot; a run that a share boundary cuts leaves its partial
//                       sum in a per-CTA piece buffer.
//   state_fixup       : every cut run's pieces summed in CTA order into its slot,
//                       so each slot has exactly one writer and one summation
//                       order: the result does not depend on the schedule.
// Every mbarrier wait is bounded; on overrun the kernel records LLA_ERR_TIMEOUT
// in the device error word, lets its own copies and MMAs land and returns.
#include "lla_tc_ptx.cuh"

namespace lla {
namespace {

constexpr int kPrepThreads = 256;
constexpr int kMaxStateTiles = 8192;  // a head's tile totals staged in shared memory

// The sequences whose state sets are built: dense (cu == nullptr: sequence bh has T rows
// starting at row bh * T) or packed (sequence b of head h, bh = b * H + h, has
// cu[b+1] - cu[b] <= T rows starting at row h * total + cu[b]; a length outside those
// bounds is recorded as bad input and the sequence treated as empty). item_off[bh] is
// the first item of sequence bh in the flattened tile list (state_offsets_kernel).
struct StateSeqs {
    const int32_t* cu;
    int T, H, total;
    const int* item_off;  // packed only
    int nte;              // dense only: items of every sequence
};

// One sequence: first row, length, last position, full tiles before the tile of pos, and
// the levels of the m virtual tiles over the tile of pos (0, then the held levels 1..7,
// four bits each).
struct SeqInfo {
    int base, len, pos, Pt, m;
    uint32_t packed;
};

// First item of sequence bh in the flattened list (bh = BH: all items).
__device__ __forceinline__ int first_item(const StateSeqs& sq, int bh) {
    return sq.cu ? sq.item_off[bh] : bh * sq.nte;
}

__device__ __forceinline__ SeqInfo seq_info(const StateSeqs& sq, int bh, int* err) {
    SeqInfo si;
    if (!sq.cu) {
        si.base = bh * sq.T;
        si.len = sq.T;
    } else {
        const int b = bh / sq.H, h = bh - b * sq.H;
        const int c0 = sq.cu[b], c1 = sq.cu[b + 1];
        if (c0 < 0 || c1 < c0 || c1 > sq.total || c1 - c0 > sq.T) {
            if (err) record_error(err, kDevBadInput);
            si.base = 0;
            si.len = 0;
        } else {
            si.base = h * sq.total + c0;
            si.len = c1 - c0;
        }
    }
    si.pos = si.len - 1;
    si.Pt = si.len > 0 ? si.pos >> 7 : 0;
    si.m = 0;
    si.packed = 0;
    if (si.len > 0) {
        si.m = 1;  // level 0 at bits 0..3
        for (int l = 1; l <= 7; l++)
            if ((si.pos >> (l - 1)) & 1) si.packed |= static_cast<uint32_t>(l) << (4 * si.m++);
    }
    return si;
}

// item_off[bh] = sum over earlier sequences of their items (full tiles + virtual tiles),
// item_off[BH] = all items. One block of 1024 threads.
__global__ void __launch_bounds__(1024) state_offsets_kernel(StateSeqs sq, int* __restrict__ item_off, int BH,
                                                             int* err) {
    __shared__ int warp_tot[32];
    __shared__ int carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int b0 = 0; b0 < BH; b0 += 1024) {
        const int bh = b0 + tid;
        int n = 0;
        if (bh < BH) {
            const SeqInfo si = seq_info(sq, bh, err);
            n = si.len > 0 ? si.Pt + si.m : 0;
        }
        int incl = n;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        int before = carry;
        for (int w = 0; w < warp; w++) before += warp_tot[w];
        if (bh < BH) item_off[bh] = before + incl - n;
        __syncthreads();
        if (tid == 1023) carry = before + incl;
        __syncthreads();
    }
    if (tid == 0) item_off[BH] = carry;
}

// g[item_off[bh] + u] = sum of log_a over full tile u of sequence bh.
// grid (ceil(max Pt / 8), BH), 256 threads: one warp per full tile.
__global__ void __launch_bounds__(256) state_tile_totals_kernel(const float* __restrict__ log_a,
                                                                float* __restrict__ g, StateSeqs sq) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int u = blockIdx.x * 8 + warp, bh = blockIdx.y;
    const SeqInfo si = seq_info(sq, bh, nullptr);
    if (u >= si.Pt) return;
    const float* a = log_a + static_cast<size_t>(si.base) + static_cast<size_t>(u) * kTile;
    float s = a[lane] + a[lane + 32] + a[lane + 64] + a[lane + 96];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) g[first_item(sq, bh) + u] = s;
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

// Slot l is held at position pos: level 0 always, level l >= 1 when bit l - 1 of pos is set.

// grid (BH, 1 + Lmax), 256 threads, dynamic shared memory: max Pt floats. Block y = 0
// scans the sequence's tile totals into tail[item_off[bh] + u]; block y = 1 + l zeroes
// slot l if it is held at pos (the MMA kernel adds into it).
__global__ void __launch_bounds__(kPrepThreads)
    state_prep_kernel(const float* __restrict__ log_a, const float* __restrict__ g, float* __restrict__ tail,
                      float* __restrict__ states, StateSeqs sq, int Lmax, int msz) {
    extern __shared__ float g_sh[];
    __shared__ float warp_tot[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int bh = blockIdx.x;
    const SeqInfo si = seq_info(sq, bh, nullptr);
    if (si.len == 0) return;  // an empty sequence holds no slot
    const int pos = si.pos, Pt = si.Pt;
    const size_t off = first_item(sq, bh);
    const int base = Pt * kTile;     // first token of the tile of pos
    const int n = pos - base + 1;    // its tokens, 1..128
    const float* a = log_a + static_cast<size_t>(si.base);

    // tail_u for every full tile, summed from pos backwards
    float ts = (tid < n) ? a[base + tid] : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ts += __shfl_xor_sync(0xffffffffu, ts, off);
    if (lane == 0) warp_tot[warp] = ts;
    __syncthreads();
    float tail_tot = 0.f;
    for (int w = 0; w < 8; w++) tail_tot += warp_tot[w];
    __syncthreads();
    for (int u = tid; u < Pt; u += kPrepThreads) g_sh[u] = g[off + u];
    __syncthreads();
    // thread t owns the tiles [hi - C, hi), hi = Pt - t C: thread 0 the newest
    const int C = (Pt + kPrepThreads - 1) / kPrepThreads;
    const int hi = Pt - tid * C;
    const int lo = hi - C > 0 ? hi - C : 0;
    float csum = 0.f;
    for (int u = hi - 1; u >= lo; u--) csum += g_sh[u];
    float run = tail_tot + block_excl_scan256(csum, warp_tot);
    for (int u = hi - 1; u >= lo; u--) {
        tail[off + u] = run;
        run += g_sh[u];
    }
}

template <int DV>
struct StateCfg {
    static constexpr int kStages = DV == 64 ? 3 : 2;
    static constexpr int kKBytes = 2 * kPanelBytes;            // K tile: 128 tokens x 128 dk
    static constexpr int kVBytes = (DV / 64) * kPanelBytes;    // V tile (scaled hi in place) / the lo part
    static constexpr int kStageBytes = kKBytes + 2 * kVBytes;
    static constexpr uint32_t kTxBytes = kKBytes + kVBytes;
    static constexpr int kBytes = kStages * kStageBytes + 1024;  // + alignment slack
    static constexpr int kThreads = 512;
    static constexpr uint32_t kAccCols = 2 * DV;               // [hi part | lo part] of one accumulator
    static constexpr uint32_t kTmemCols = 2 * kAccCols;        // two accumulators
};

// Slot of tile u of a head: a full tile (u < Pt) sits at level 8 + floor(log2(u xor Pt));
// tile Pt + j is the j-th virtual tile over the tile of pos.
__device__ __forceinline__ int tile_level(int u, int Pt, uint32_t tail_lev) {
    return u < Pt ? 8 + 31 - __clz(u ^ Pt) : static_cast<int>((tail_lev >> (4 * (u - Pt))) & 15u);
}

// 512 threads: warp 0 TMA producer, warp 1 TMEM owner + MMA issuer, warps 4..11
// scale V (two threads per token row, four 16-byte chunks of each 128-byte panel
// row each; every warp derives the tile's decay prefix on its own, so the scaler
// warps never wait for one another), warps 12..15 drain accumulators (TMEM lane quadrant = warp % 4, one
// dk row per thread). Sequence bh contributes Pt + m tiles to the flattened list,
// starting at item_off[bh]; the CTAs take equal shares of item_off[BH] items.
template <int DV>
__global__ void __launch_bounds__(512, 1)
    tc_state_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const float* __restrict__ log_a, const float* __restrict__ tail, float* __restrict__ states,
                    StateSeqs sq, int BH, int Lmax, float* __restrict__ pieces, int* __restrict__ piece_slot,
                    int* __restrict__ piece_flags, int* err) {
    using C = StateCfg<DV>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full_bar[S], scaled_bar[S], empty_bar[S], acc_full[2], acc_empty[2], drain_bar;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int fail_sh;

    grid_dep_wait();  // the item offsets and tails (launched early, see launch_pdl)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int total = first_item(sq, BH);
    const int t0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * total / gridDim.x);
    const int t1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * total / gridDim.x);
    volatile int* fail = &fail_sh;

    if (tid == 0) {
        for (int s = 0; s < S; s++) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&scaled_bar[s], 8);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        mbar_init(&drain_bar, 1);
        fence_mbar_init();
        fail_sh = 0;
        // this share's pieces: none yet (bit 2 marks a share without items)
        piece_slot[2 * blockIdx.x] = piece_slot[2 * blockIdx.x + 1] = -1;
        piece_flags[2 * blockIdx.x] = t0 == t1 ? 4 : 0;
        piece_flags[2 * blockIdx.x + 1] = 0;
    }
    if (warp == 1) tmem_alloc(&tmem_base_sh, C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    auto fail_now = [&]() {
        if (atomicExch(&fail_sh, 1) == 0) record_error(err, kDevTimeout);
    };
    // Walk of this CTA's tiles without divisions: sequence bh (and its SeqInfo), tile u of
    // it, its slot, and whether the next tile (f + 1 < t1) continues the same run.
    struct Cursor {
        int bh, u, lvl;
        SeqInfo si;
        bool last_of_run;
    };
    auto cursor_at = [&](int f) {
        Cursor c;
        // the sequence whose item range holds f: the last bh with first_item(bh) <= f
        int lo = 0, hi = BH;
        if (!sq.cu) {
            lo = f / sq.nte < BH ? f / sq.nte : BH - 1;
        } else {
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (sq.item_off[mid] <= f) lo = mid; else hi = mid;
            }
        }
        c.bh = lo;
        c.si = seq_info(sq, lo, nullptr);
        c.u = f - first_item(sq, lo);
        c.lvl = tile_level(c.u, c.si.Pt, c.si.packed);
        c.last_of_run = true;
        return c;
    };
    // advances c from tile f to f + 1 and fills c.last_of_run for tile f
    auto step = [&](Cursor& c, int f) {
        Cursor n = c;
        n.u++;
        if (n.u >= n.si.Pt + n.si.m) {
            // next sequence with tiles (empty ones have none); stays in range while f + 1 < t1
            n.u = 0;
            do {
                n.bh++;
                n.si = seq_info(sq, n.bh < BH ? n.bh : BH - 1, nullptr);
            } while (n.bh < BH - 1 && n.si.len == 0);
        }
        n.lvl = tile_level(n.u, n.si.Pt, n.si.packed);
        c.last_of_run = (f + 1 >= t1) || n.bh != c.bh || n.lvl != c.lvl;
        n.last_of_run = true;
        return n;
    };

    int issued = 0;  // producer: tiles whose copies were issued
    if (warp == 0) {
        if (lane == 0) {
            Cursor c = cursor_at(t0);
            int s = 0;
            uint32_t ph = 0;
            for (int f = t0; f < t1 && !*fail; f++, issued++) {
                if (f - t0 >= S && !mbar_wait(&empty_bar[s], ph ^ 1u)) {
                    fail_now();
                    break;
                }
                // rows of the tile of pos past the sequence's end are another sequence's
                // (weight 0) or past the tensor (filled with zeros)
                const int r0 = c.si.base + (c.u < c.si.Pt ? c.u : c.si.Pt) * kTile;
                uint8_t* st = smem + s * C::kStageBytes;
                mbar_expect_tx(&full_bar[s], C::kTxBytes);
                tma_load_2d(st, &tm_k, &full_bar[s], 0, r0);
                tma_load_2d(st + kPanelBytes, &tm_k, &full_bar[s], 64, r0);
#pragma unroll
                for (int p = 0; p < DV / 64; p++)
                    tma_load_2d(st + C::kKBytes + p * kPanelBytes, &tm_v, &full_bar[s], 64 * p, r0);
                c = step(c, f);
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // A = K^T (MN-major); B = [hi | lo] of w o V (MN-major, N = 2 DV: the lo panels follow the
            // hi panels at the same 16 KB panel stride), so one MMA per 16-token step covers both parts
            constexpr uint32_t kIdesc = idesc_bf16(kDk, 2 * DV, 1, 1);
            // a K step of 16 tokens moves every operand by 2048 B: +128 in the descriptor's address field
            const uint64_t kdesc0 = sdesc(smem_u32(smem), kPanelBytes, 1024);
            const uint64_t vdesc0 = sdesc(smem_u32(smem + C::kKBytes), kPanelBytes, 1024);
            constexpr uint64_t kStageStep = C::kStageBytes >> 4;
            Cursor c = cursor_at(t0);
            bool starting = true;
            int run = 0, s = 0;
            uint32_t ph = 0;
            for (int f = t0; f < t1 && !*fail; f++) {
                const Cursor nc = step(c, f);
                const bool ending = c.last_of_run;
                const int buf = run & 1;
                if (starting && run >= 2 && !mbar_wait(&acc_empty[buf], ((run >> 1) - 1) & 1)) {
                    fail_now();
                    break;
                }
                if (!mbar_wait(&scaled_bar[s], ph)) {
                    fail_now();
                    break;
                }
                tc_fence_after();
                const uint64_t so = kStageStep * s;
                const uint32_t d = tmem + buf * C::kAccCols;
#pragma unroll
                for (int kk = 0; kk < kTile / 16; kk++) {
                    const uint64_t ko = so + 128u * kk;
                    mma_bf16(d, kdesc0 + ko, vdesc0 + ko, kIdesc, (starting && kk == 0) ? 0u : 1u);
                }
                mma_commit(&empty_bar[s]);
                if (ending) {
                    mma_commit(&acc_full[buf]);
                    run++;
                }
                starting = ending;
                c = nc;
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            // every MMA issued above has completed before TMEM and shared memory go away
            mma_commit(&drain_bar);
            if (!mbar_wait(&drain_bar, 0)) fail_now();
        }
    } else if (warp >= 4 && warp < 12) {
        const int sidx = tid - 128;
        const int row = sidx & 127, half = sidx >> 7, w4 = (warp - 4) & 3;
        // log_a of the tile's tokens 32 j + lane (0 past pos), j = 0..3, and the tile's tail decay
        auto tile_inputs = [&](const Cursor& c, float* la, float& tlv) {
            const size_t hb = static_cast<size_t>(c.si.base);
            if (c.u < c.si.Pt) {
#pragma unroll
                for (int j = 0; j < 4; j++) la[j] = log_a[hb + static_cast<size_t>(c.u) * kTile + 32 * j + lane];
                tlv = tail[first_item(sq, c.bh) + c.u];
            } else {
                const int first = c.si.Pt * kTile, n_last = c.si.pos - first + 1;  // the tile of pos
#pragma unroll
                for (int j = 0; j < 4; j++) la[j] = 32 * j + lane < n_last ? log_a[hb + first + 32 * j + lane] : 0.f;
                tlv = 0.f;
            }
        };
        // inputs are fetched two tiles ahead
        Cursor c0 = cursor_at(t0);
        Cursor c1 = step(c0, t0);
        float la0[4] = {0.f, 0.f, 0.f, 0.f}, la1[4], tl0 = 0.f, tl1 = 0.f;
        if (t0 < t1) tile_inputs(c0, la0, tl0);
        if (t0 + 1 < t1) tile_inputs(c1, la1, tl1);
        int s = 0;
        uint32_t ph = 0;
        for (int f = t0; f < t1; f++) {
            if (__any_sync(0xffffffffu, *fail != 0)) break;
            const int u = c0.u;
            const SeqInfo si = c0.si;
            float x[4];
#pragma unroll
            for (int j = 0; j < 4; j++) x[j] = la0[j];
            const float tlv = tl0;
            // advance the queue: c0 <- c1, c1 <- tile f + 2
            c0 = c1;
#pragma unroll
            for (int j = 0; j < 4; j++) la0[j] = la1[j];
            tl0 = tl1;
            if (f + 1 < t1) {
                c1 = step(c1, f + 1);
                if (f + 2 < t1) tile_inputs(c1, la1, tl1);
            }
            // in-tile inclusive prefix of log_a: four 32-token warp scans
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    const float y = __shfl_up_sync(0xffffffffu, x[j], off);
                    if (lane >= off) x[j] += y;
                }
            }
            float before = 0.f, tot = 0.f;
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const float cj = __shfl_sync(0xffffffffu, x[j], 31);
                before += (j < w4) ? cj : 0.f;
                tot += cj;
            }
            const float incl = before + (w4 == 0 ? x[0] : w4 == 1 ? x[1] : w4 == 2 ? x[2] : x[3]);
            // decay from token row to pos: the rest of the tile, then the tail
            float w = exp2f((tlv + tot - incl) * kLog2e);
            if (u >= si.Pt) {
                // virtual tile: only the keys of its level, none past pos
                const int first = si.Pt * kTile;
                const bool keep = row < si.pos - first + 1 &&
                                  fenwick_level(si.pos, first + row) == tile_level(u, si.Pt, si.packed);
                w = keep ? w : 0.f;
            }
            const int cs = s;
            const uint32_t cph = ph;
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
            if (!warp_wait(&full_bar[cs], cph)) {
                if (lane == 0) fail_now();
                break;
            }
            uint8_t* vrow = smem + cs * C::kStageBytes + C::kKBytes + row * 128;
#pragma unroll
            for (int p = 0; p < DV / 64; p++) {
#pragma unroll
                for (int c = half * 4; c < half * 4 + 4; c++) {
                    const uint32_t off = p * kPanelBytes + ((c ^ (row & 7)) << 4);
                    uint4* hp = reinterpret_cast<uint4*>(vrow + off);
                    uint4* lp = reinterpret_cast<uint4*>(vrow + C::kVBytes + off);
                    const uint4 xv = *hp;
                    const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
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
            if (lane == 0) mbar_arrive(&scaled_bar[cs]);
        }
    } else if (warp >= 12) {
        const int quad = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        int run = 0;
        Cursor c = cursor_at(t0);
        // whether this share's first run continues the previous share's last run
        bool cut_start = false;
        if (t0 > 0 && t0 < t1) {
            const Cursor pc = cursor_at(t0 - 1);
            cut_start = pc.bh == c.bh && pc.lvl == c.lvl;
        }
        for (int f = t0; f < t1; f++) {
            const Cursor nc = step(c, f);
            const Cursor cur = c;
            c = nc;
            if (!cur.last_of_run) continue;
            const int buf = run & 1;
            if (*fail) break;
            if (!warp_wait(&acc_full[buf], (run >> 1) & 1)) {
                if (lane == 0) fail_now();
                break;
            }
            tc_fence_after();
            const int bh = cur.bh, l = cur.lvl;
            // a run held whole by this share is the slot's only writer; a cut one leaves a piece
            const bool cs = run == 0 && cut_start;
            const bool ce = f + 1 == t1 && t1 < total && nc.bh == cur.bh && nc.lvl == cur.lvl;
            float* slot;  // row 0 of the dk x DV slot (or piece) this run is drained into
            if (!cs && !ce) {
                slot = states + (static_cast<size_t>(bh) * Lmax + l) * kDk * DV;
            } else {
                const int kind = cs ? 0 : 1;
                slot = pieces + static_cast<size_t>(2 * blockIdx.x + kind) * kDk * DV;
                if (warp == 12 && lane == 0) {
                    piece_slot[2 * blockIdx.x + kind] = bh * Lmax + l;
                    piece_flags[2 * blockIdx.x + kind] = (cs ? 1 : 0) | (ce ? 2 : 0);
                }
            }
#pragma unroll
            for (int c0 = 0; c0 < DV; c0 += 32) {
                float x[32], y[32];
                tmem_ld32(tmem + lane_base + buf * C::kAccCols + c0, x);
                tmem_ld32(tmem + lane_base + buf * C::kAccCols + DV + c0, y);
                // 16-byte chunks of this row, transposed within lane groups so that each store
                // writes 64 contiguous bytes of 8 rows (row quad * 32 + (lane & ~3) + i)
#pragma unroll
                for (int hh = 0; hh < 2; hh++) {
                    uint4 ch[4];
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const int e = 16 * hh + 4 * j;
                        ch[j] = make_uint4(__float_as_uint(x[e] + y[e]), __float_as_uint(x[e + 1] + y[e + 1]),
                                           __float_as_uint(x[e + 2] + y[e + 2]), __float_as_uint(x[e + 3] + y[e + 3]));
                    }
                    lane_group_transpose(ch, lane);
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const int r = quad * 32 + (lane & ~3) + i;
                        *reinterpret_cast<uint4*>(slot + static_cast<size_t>(r) * DV + c0 + 16 * hh + 4 * (lane & 3)) = ch[i];
                    }
                }
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

// One block per tc_state share b: if b's last run continues into the next share and began in b
// (b leads that run), the run's pieces are summed in share order -- b's piece, then the first
// piece of each following share while the run continues (shares without items skipped) -- and
// stored into the run's slot. 256 threads, float4 elements of the dk x dv slot.
__global__ void __launch_bounds__(256) state_fixup_kernel(const float* __restrict__ pieces,
                                                          const int* __restrict__ piece_slot,
                                                          const int* __restrict__ piece_flags, float* __restrict__ states,
                                                          int n_shares, int msz) {
    grid_dep_wait();  // tc_state's pieces (launched early, see launch_pdl)
    const int b = blockIdx.x;
    int k = -1;
    if (piece_flags[2 * b + 1] & 2) k = 1;
    else if ((piece_flags[2 * b] & 6) == 2) k = 0;
    if (k < 0 || (piece_flags[2 * b + k] & 1)) return;  // no run leaves b, or b only continues one
    float4* dst = reinterpret_cast<float4*>(states + static_cast<size_t>(piece_slot[2 * b + k]) * msz);
    const float4* first = reinterpret_cast<const float4*>(pieces + static_cast<size_t>(2 * b + k) * msz);
    for (int e = threadIdx.x; e < msz / 4; e += blockDim.x) {
        float4 acc = first[e];
        for (int c = b + 1; c < n_shares; c++) {
            const int fl = piece_flags[2 * c];
            if (fl & 4) continue;  // a share without items
            const float4 x = reinterpret_cast<const float4*>(pieces + static_cast<size_t>(2 * c) * msz)[e];
            acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
            if (!(fl & 2)) break;  // the run ends in share c
        }
        dst[e] = acc;
    }
}

// CTAs of tc_state: one per SM (the item count is only known on the device).
int state_shares() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
        cudaGetLastError();
        sms = 152;
    }
    return sms < 1024 ? sms : 1024;
}

// Workspace: item offsets | tile totals g | tails | pieces [shares][2][dk][dv] | piece slots, flags.
size_t state_base_bytes(size_t BH, int T) {
    return (static_cast<size_t>(BH + 1) * sizeof(int) + 255) / 256 * 256 +
           (2 * BH * ((static_cast<size_t>(T - 1) >> 7) + 8) * sizeof(float) + 255) / 256 * 256;
}

template <int DV>
cudaError_t tc_prefill_state_dv(const void* k, const void* v, const float* log_a, float* states, int BH, int H,
                                int T, int Lmax, void* workspace, int* err, cudaStream_t stream, const int32_t* cu,
                                int total) {
    const int maxPt = (T - 1) >> 7;
    const size_t off_bytes = (static_cast<size_t>(BH + 1) * sizeof(int) + 255) / 256 * 256;
    int* item_off = static_cast<int*>(workspace);
    float* g = reinterpret_cast<float*>(static_cast<char*>(workspace) + off_bytes);
    float* tail = g + static_cast<size_t>(BH) * (maxPt + 8);
    const int sms = state_shares();
    float* pieces = reinterpret_cast<float*>(static_cast<char*>(workspace) + state_base_bytes(BH, T));
    int* piece_slot = reinterpret_cast<int*>(pieces + static_cast<size_t>(2) * sms * kDk * DV);
    int* piece_flags = piece_slot + 2 * sms;
    int nte = 0;  // dense: every sequence has the same items
    if (!cu) {
        const int pos = T - 1;
        nte = (pos >> 7) + 1;
        for (int l = 1; l <= 7; l++) nte += (pos >> (l - 1)) & 1;
    }
    const StateSeqs sq{cu, T, H, total, item_off, nte};
    if (cu) state_offsets_kernel<<<1, 1024, 0, stream>>>(sq, item_off, BH, err);
    if (maxPt > 0) {
        state_tile_totals_kernel<<<dim3((maxPt + 7) / 8, BH), 256, 0, stream>>>(log_a, g, sq);
        note_launch(stream, "state_tile_totals");
    }
    {
        const size_t smem = static_cast<size_t>(maxPt) * sizeof(float);
        cudaError_t e = cudaFuncSetAttribute(state_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        state_prep_kernel<<<BH, kPrepThreads, smem, stream>>>(log_a, g, tail, states, sq, Lmax, kDk * DV);
        note_launch(stream, "state_prep");
    }
    {
        CUtensorMap tk, tv;
        const uint64_t rows = cu ? static_cast<uint64_t>(H) * total : static_cast<uint64_t>(BH) * T;
        if (!make_map(&tk, k, rows, kDk) || !make_map(&tv, v, rows, DV)) return cudaErrorInvalidValue;
        using C = StateCfg<DV>;
        cudaError_t e = cudaFuncSetAttribute(tc_state_kernel<DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kBytes);
        if (e != cudaSuccess) return e;
        // the item count is only known on the device: one CTA per SM, each takes its share
        e = launch_pdl(tc_state_kernel<DV>, dim3(sms), dim3(C::kThreads), C::kBytes, stream, tk, tv, log_a,
                       static_cast<const float*>(tail), states, sq, BH, Lmax, pieces, piece_slot, piece_flags, err);
        if (e != cudaSuccess) return e;
        note_launch(stream, "tc_state");
        e = launch_pdl(state_fixup_kernel, dim3(sms), dim3(256), 0, stream, static_cast<const float*>(pieces),
                       static_cast<const int*>(piece_slot), static_cast<const int*>(piece_flags), states, sms,
                       kDk * DV);
        if (e != cudaSuccess) return e;
        note_launch(stream, "state_fixup");
    }
    return cudaGetLastError();
}

}  // namespace

bool tc_state_supported(int dtype, int dk, int dv, int B, int H, int T) {
    const int64_t Pt = (static_cast<int64_t>(T) - 1) >> 7;
    // (the tensor maps want at least one 128-row box of rows)
    return dtype == 0 && dk == kDk && (dv == 64 || dv == 128) && Pt <= kMaxStateTiles &&
           static_cast<int64_t>(B) * H * T >= kTile &&
           static_cast<int64_t>(B) * H * (Pt + 8) < (int64_t(1) << 31) &&
           static_cast<int64_t>(B) * H * T < (int64_t(1) << 31);
}

bool tc_state_supported_packed(int dtype, int dk, int dv, int n_seq, int H, int total, int max_T) {
    const int64_t Pt = (static_cast<int64_t>(max_T) - 1) >> 7;
    return dtype == 0 && dk == kDk && (dv == 64 || dv == 128) && Pt <= kMaxStateTiles &&
           static_cast<int64_t>(H) * total >= kTile && static_cast<int64_t>(H) * total < (int64_t(1) << 31) &&
           static_cast<int64_t>(n_seq) * H * (Pt + 8) < (int64_t(1) << 31);
}

size_t tc_state_workspace_bytes(int B, int H, int T, int dv) {
    const size_t sms = static_cast<size_t>(state_shares());
    return state_base_bytes(static_cast<size_t>(B) * H, T) + 2 * sms * kDk * dv * sizeof(float) +
           4 * sms * sizeof(int) + 256;
}

cudaError_t tc_prefill_state(const void* k, const void* v, const float* log_a, float* states, int B, int H, int T,
                             int dv, int Lmax, void* workspace, int* err, cudaStream_t stream, const int32_t* cu,
                             int total) {
    if (dv == 64)
        return tc_prefill_state_dv<64>(k, v, log_a, states, B * H, H, T, Lmax, workspace, err, stream, cu, total);
    return tc_prefill_state_dv<128>(k, v, log_a, states, B * H, H, T, Lmax, workspace, err, stream, cu, total);
}

}  // namespace lla
