// Tensor-core (tcgen05 / TMEM / TMA) path of log-linear Mamba-2 attention
// prefill, bf16 q/k/v with fp32 accumulation, dk in {64, 128}, dv in {64, 128},
// T % 128 == 0. dk = 64 runs the dk = 128 kernels on zero-padded operands: the
// tensor maps of q and k have the real 64 columns, so the second 64-column panel
// of every Q and K tile lies wholly outside the tensor and TMA fills it with
// zeros; every product over dk is then the 64-column one, and the Fenwick nodes
// (128 x dv) carry zero rows 64..127.
//
// Chunkwise algorithm ("Log-Linear Attention", pt §2 "Forma Recorrente e
// Paralela" / fr §2 "Algorithmes Efficaces": dense intra-block work,
// hierarchical inter-block state passing, O(T log T), matmul-rich) laid out
// on 128-token tiles (the M = 128 tcgen05 shape). Tile j covers tokens
// [128 j, 128 j + 128). Within a tile, every key s <= t is handled densely
// with its exact Fenwick level 1 + floor(log2(t xor s)) <= 7. A key in an
// earlier tile i sits at level 8 + floor(log2(j xor i)), and the keys of level
// 8 + p are exactly the tiles of the aligned block ((j >> p) - 1) << p ..
// ((j >> p) << p) - 1, present when bit p of j is set. That block's decayed
// state sum is the Fenwick node (p, m = (j >> p) - 1): a dk x dv matrix.
//
// Kernels (one stream, in order):
//   tc_nodes  : per (head, segment of 2^q tiles): S_u = K_u^T diag(w) V_u on
//               tcgen05 (w_s = decay from s to the tile end), then the level
//               accumulators A_l <- e^{g_u} A_l + S_u kept in TMEM; a node is
//               written (bf16) when its block closes. Also writes the tile
//               log-decay totals g_u and each full segment's fp32 total.
//   tc_merge  : levels above a segment: fp32 pyramid over segment totals
//               (SIMT, small), writing the nodes that are read (bf16).
//   tc_output : per (head, tile): S = Q K^T (tcgen05, TMEM), masked with
//               decay and lambda into bf16 P (smem), O = P V plus, per set
//               bit p of j, L_p = Q B_p (tcgen05, TMEM); epilogue
//               O + sum_p lambda_t^(8+p) exp(decay) L_p -> bf16.
// Only even-indexed nodes are ever read (node (p, m) is read by tile j iff
// j >> p == m + 1, and bit p of j is set), so only those are stored.
//
// Every mbarrier wait is bounded: on overrun a kernel records
// LLA_ERR_TIMEOUT in the device error word, waits (bounded) for its own
// in-flight work, frees its TMEM and returns.
#include "lla_tc_ptx.cuh"

namespace lla {

// Failure-path test hooks of tc_output_pp (set from the host by tc_set_debug_waits):
// the bound, in SM cycles, on the kernel's pipeline waits (its drain waits, which let
// in-flight copies and MMAs land, always keep the full bound), and a switch that makes
// the epilogue first wait on a barrier nothing arrives at, so that wait runs out.
__device__ long long tc_pipe_wait_limit = 4000000000LL;
__device__ int tc_debug_hold = 0;

namespace {

struct LevelOffsets { int off[32]; };

// Where a head's rows are. Dense layout (seq == nullptr): head bh = b * H + h is rows bh * T ..
// of every [B*H*T, .] tensor. Packed variable-length sequences: the tensors are [H, total_T, .]
// and sequence i owns rows seq[i].x .. seq[i].x + seq[i].y - 1 of every head (a validated copy of
// cu_seqlens); the workspace keeps the dense layout with T = the longest sequence rounded up to
// a tile, head bh = i * H + h.
struct SeqMap {
    const int2* seq;          // per sequence {first row, length}; null: dense
    const int* tile_prefix;   // [n_seq + 1]: H x (tiles of the sequences before i)
    int H, n_seq, total_T;
};

// First input row and length of head bh.
__device__ __forceinline__ void seq_of(const SeqMap& sm, int bh, int T, int& rowbase, int& len) {
    if (!sm.seq) {
        rowbase = bh * T;
        len = T;
        return;
    }
    const int i = bh / sm.H, h = bh - i * sm.H;
    const int2 s = sm.seq[i];
    rowbase = h * sm.total_T + s.x;
    len = s.y;
}

// One block: the validated sequence table and the tile prefix of the packed layout. A sequence
// whose bounds are inconsistent (negative start, decreasing offsets, rows past total_T, longer
// than max_T) is recorded as bad input and gets length 0 (no tiles, no output rows written).
__global__ void __launch_bounds__(1024) seq_table_kernel(const int32_t* __restrict__ cu, int2* __restrict__ seq,
                                                         int* __restrict__ tile_prefix, int n_seq, int H, int total_T,
                                                         int max_T, int* err) {
    __shared__ int part[1024];
    const int tid = threadIdx.x;
    const int per = (n_seq + 1023) / 1024;
    const int i0 = tid * per, i1 = min(n_seq, i0 + per);
    int sum = 0;
    for (int i = i0; i < i1; i++) {
        const int c0 = cu[i], c1 = cu[i + 1];
        const bool ok = c0 >= 0 && c1 >= c0 && c1 <= total_T && c1 - c0 <= max_T;
        if (!ok) record_error(err, kDevBadInput);
        const int len = ok ? c1 - c0 : 0;
        seq[i] = make_int2(ok ? c0 : 0, len);
        sum += (len + kTile - 1) / kTile;
    }
    part[tid] = sum;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int t = 0; t < 1024; t++) {
            const int x = part[t];
            part[t] = run;
            run += x;
        }
    }
    __syncthreads();
    int run = part[tid];
    for (int i = i0; i < i1; i++) {
        tile_prefix[i] = H * run;
        run += (seq[i].y + kTile - 1) / kTile;
    }
    if (i1 == n_seq && i0 < i1) tile_prefix[n_seq] = H * run;
    if (n_seq == 0 && tid == 0) tile_prefix[0] = 0;
}

// ------------------------------------------------------------------ tc_nodes

template <int DV>
struct NodesSmem {
    static constexpr int kKBytes = 2 * kPanelBytes;             // K tile: 128 tokens x 128 dk
    static constexpr int kVBytes = (DV / 64) * kPanelBytes;     // V tile: 128 tokens x DV
    static constexpr int kStageBytes = kKBytes + kVBytes;
    static constexpr int kStages = 2;
    static constexpr int kBytes = kStages * kStageBytes + 1024;  // + alignment slack
};

// grid (num_segments, B*H), 256 threads: two threads per dk row (= TMEM lane), each
// owning half of the dv columns. Segment s covers tiles [s 2^Q, (s+1) 2^Q).
// Per tile u: S_u = K_u^T diag(w) V_u on tcgen05 into TMEM buffer u % 2 (the MMA of
// tile u+1 runs while tile u's epilogue reads its buffer); then, in registers,
// A_l <- e^{g_u} A_l + S_u for the levels l = 1..Q whose blocks contain u. A block
// that closes at u is written out as a node (bf16) when it is read by a later tile,
// and the level-Q block (the whole segment) as the segment's fp32 total.
template <int DV, int Q>
__global__ void __launch_bounds__(256, 2)
    tc_nodes_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const float* __restrict__ log_a, float* __restrict__ g_tiles, __nv_bfloat16* __restrict__ nodes,
                    float* __restrict__ seg_tot, float* __restrict__ tok_cl2, float* __restrict__ tok_colw, int T,
                    int NT, int node_count, const __grid_constant__ LevelOffsets lo, const SeqMap sm,
                    int* __restrict__ tile_counter, int* err) {
    constexpr int DH = DV / 2;  // columns per thread
    constexpr int kSegTiles = 1 << Q;
    using S = NodesSmem<DV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar_full[2], bar_mma[2];
    __shared__ uint32_t tmem_base_sh;
    __shared__ float warp_tot[8];
    __shared__ float cl2_sh[kSegTiles][kTile];  // in-tile decay prefix, log2 units
    __shared__ float g2_sh[kSegTiles];          // tile totals, log2 units
    __shared__ int fail_sh;

    grid_dep_launch();  // the merge kernel may be launched while this grid drains
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // the output kernel's tile counter: it starts claiming tiles only after this grid has
    // completed (its launch waits on the merge kernel, which waits on this one)
    if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) *tile_counter = 0;
    const int seg = blockIdx.x, bh = blockIdx.y;
    const int tile0 = seg * kSegTiles;
    int rowbase, len;
    seq_of(sm, bh, T, rowbase, len);
    const int NTi = (len + kTile - 1) / kTile;  // this head's tiles (NT in the dense layout)
    const int ntiles = min(kSegTiles, NTi - tile0);
    if (ntiles <= 0) return;  // packed layout: past this sequence's last tile
    const int row = tid & 127;         // dk row in the epilogue, token row while scaling V
    const int half = tid >> 7;         // which half of the dv columns / of the V row
    const int quad = warp & 3;         // TMEM lane quadrant of this warp
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    constexpr uint32_t kTxBytes = S::kStageBytes;
    constexpr uint32_t kCols = 2 * DV <= 32 ? 32 : 2 * DV;

    if (tid == 0) {
        for (int b = 0; b < 2; b++) {
            mbar_init(&bar_full[b], 1);
            mbar_init(&bar_mma[b], 1);
        }
        fence_mbar_init();
        fail_sh = 0;
    }
    if (warp == 0) tmem_alloc(&tmem_base_sh, kCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    auto stage_ptr = [&](int s) { return smem + s * S::kStageBytes; };
    auto issue_tile = [&](int u) {
        const int s = u & 1;
        uint8_t* st = stage_ptr(s);
        const int r0 = rowbase + (tile0 + u) * kTile;
        mbar_expect_tx(&bar_full[s], kTxBytes);
        // K and V are read again only by the output kernel, after every node kernel: keeping them
        // in L2 would only push out the segment totals and nodes that are read back sooner
        const uint64_t pol = l2_evict_first();
        tma_load_2d_hint(st, &tm_k, &bar_full[s], 0, r0, pol);
        tma_load_2d_hint(st + kPanelBytes, &tm_k, &bar_full[s], 64, r0, pol);
#pragma unroll
        for (int p = 0; p < DV / 64; p++)
            tma_load_2d_hint(st + S::kKBytes + p * kPanelBytes, &tm_v, &bar_full[s], 64 * p, r0, pol);
    };
    if (tid == 0) {
        issue_tile(0);
        if (ntiles > 1) issue_tile(1);
    }

    // decays of the whole segment: per tile an inclusive prefix over its 128 tokens
    // (threads 0..127, one token each), stored for the output kernel as well; every
    // tile's log_a is loaded before the first scan
    float la[kSegTiles];
#pragma unroll
    for (int u = 0; u < kSegTiles; u++) {
        const int pos = (tile0 + u) * kTile + row;
        la[u] = (half == 0 && u < ntiles && pos < len) ? log_a[static_cast<size_t>(rowbase) + pos] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kSegTiles; u++) {
        if (u >= ntiles) break;
        const size_t tok = static_cast<size_t>(bh) * T + static_cast<size_t>(tile0 + u) * kTile + row;
        float x = la[u];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        if (half == 0) {
            float base = 0.f;
            for (int w = 0; w < quad; w++) base += warp_tot[w];
            cl2_sh[u][row] = (x + base) * kLog2e;
            if (row == kTile - 1) {
                g2_sh[u] = (x + base) * kLog2e;
                g_tiles[static_cast<size_t>(bh) * NT + tile0 + u] = x + base;
            }
        }
        __syncthreads();
        if (half == 0) {
            tok_cl2[tok] = cl2_sh[u][row];
            tok_colw[tok] = exp2f(cl2_sh[u][row | 31] - cl2_sh[u][row]);
        }
    }

    constexpr uint32_t kIdesc = idesc_bf16(kDk, DV, 1, 1);  // A = K^T (MN-major), B = V (MN-major)
    const size_t msz = static_cast<size_t>(kDk) * DV;
    bool ok = true;

    // scale V rows of tile u by their decay to the tile end, then issue its MMA
    auto scale_and_mma = [&](int u) {
        const int s = u & 1;
        if (!mbar_wait(&bar_full[s], (u >> 1) & 1)) {
            ok = false;
            atomicExch(&fail_sh, 1);
        }
        __syncthreads();
        if (fail_sh) return;
        const float w = exp2f(g2_sh[u] - cl2_sh[u][row]);
        uint8_t* vbase = stage_ptr(s) + S::kKBytes;
        // this thread scales four of the eight 16-byte chunks of its token's 128-byte panel
        // row; the chunks sit in swizzled order (chunk c at c ^ (row & 7)), which also
        // spreads the lanes of a warp over all banks
#pragma unroll
        for (int p = 0; p < DV / 64; p++) {
            uint8_t* rowp = vbase + p * kPanelBytes + row * 128;
#pragma unroll
            for (int c = 0; c < 4; c++) {
                uint4* cp = reinterpret_cast<uint4*>(rowp + (((half * 4 + c) ^ (row & 7)) << 4));
                uint4 x = *cp;
                float2 f0 = unpack_bf16(x.x), f1 = unpack_bf16(x.y), f2 = unpack_bf16(x.z), f3 = unpack_bf16(x.w);
                x.x = pack_bf16(f0.x * w, f0.y * w);
                x.y = pack_bf16(f1.x * w, f1.y * w);
                x.z = pack_bf16(f2.x * w, f2.y * w);
                x.w = pack_bf16(f3.x * w, f3.y * w);
                *cp = x;
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            const uint32_t kb = smem_u32(stage_ptr(s));
            const uint32_t vb = kb + S::kKBytes;
#pragma unroll
            for (int kk = 0; kk < kTile / 16; kk++) {
                const uint64_t ad = sdesc(kb + kk * 2048, kPanelBytes, 1024);
                const uint64_t bd = sdesc(vb + kk * 2048, kPanelBytes, 1024);
                mma_bf16(tmem + s * DV, ad, bd, kIdesc, kk > 0 ? 1u : 0u);
            }
            mma_commit(&bar_mma[s]);
        }
    };

    float acc[Q > 0 ? Q : 1][DH];
    scale_and_mma(0);
    int u = 0;
    for (; u < ntiles && !fail_sh; u++) {
        const int s = u & 1;
        const int tile = tile0 + u;
        if (u + 1 < ntiles) scale_and_mma(u + 1);
        if (fail_sh) break;
        if (!mbar_wait(&bar_mma[s], (u >> 1) & 1)) {
            ok = false;
            atomicExch(&fail_sh, 1);
        }
        tc_fence_after();
        // stage s is free again: prefetch tile u + 2 into it
        if (tid == 0 && u + 2 < ntiles && ok) issue_tile(u + 2);

        float sv[DH];
#pragma unroll
        for (int c0 = 0; c0 < DH; c0 += 32) tmem_ld32(tmem + lane_base + s * DV + half * DH + c0, sv + c0);
        const float ge = exp2f(g2_sh[u]);
        // A thread holds DH consecutive values of one row (its TMEM lane); stored as they are,
        // every 16-byte store of a warp would touch 32 rows. The four lanes of a group swap
        // their 16-byte chunks (a 4 x 4 transpose, two xor-shuffle stages), so that in store i
        // the group writes row 4 g + i whole: 8 rows of 64 contiguous bytes per warp store.
        auto store_rows = [&](uint8_t* base, size_t row_stride, uint4 (&x)[4]) {
            const int c = lane & 3;
            lane_group_transpose(x, lane);
            const int r0 = (row & ~31) + (lane & ~3);
#pragma unroll
            for (int i = 0; i < 4; i++)
                *reinterpret_cast<uint4*>(base + static_cast<size_t>(r0 + i) * row_stride + 16 * c) = x[i];
        };
        auto store_node = [&](int l, int m, const float* v) {
            uint8_t* dst = reinterpret_cast<uint8_t*>(nodes + (static_cast<size_t>(bh) * node_count + lo.off[l] + (m >> 1)) * msz +
                                                      half * DH);
#pragma unroll
            for (int b = 0; b < DH / 32; b++) {  // columns [32 b, 32 b + 32) of this thread's DH
                uint4 x[4];
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    const float* w = v + 32 * b + 8 * c;
                    x[c] = make_uint4(pack_bf16(w[0], w[1]), pack_bf16(w[2], w[3]), pack_bf16(w[4], w[5]),
                                      pack_bf16(w[6], w[7]));
                }
                store_rows(dst + 64 * b, DV * sizeof(__nv_bfloat16), x);
            }
        };
        auto store_seg = [&](const float* v) {
            uint8_t* dst = reinterpret_cast<uint8_t*>(seg_tot + (static_cast<size_t>(bh) * ((NT + kSegTiles - 1) / kSegTiles) + seg) * msz +
                                                      half * DH);
#pragma unroll
            for (int hh = 0; hh < DH / 16; hh++) {  // columns [16 hh, 16 hh + 16) of this thread's DH
                uint4 x[4];
#pragma unroll
                for (int c = 0; c < 4; c++)
                    x[c] = make_uint4(__float_as_uint(v[16 * hh + 4 * c]), __float_as_uint(v[16 * hh + 4 * c + 1]),
                                      __float_as_uint(v[16 * hh + 4 * c + 2]), __float_as_uint(v[16 * hh + 4 * c + 3]));
                store_rows(dst + 64 * hh, DV * sizeof(float), x);
            }
        };
        // level 0: the tile itself
        if ((tile & 1) == 0 && tile + 1 < NTi) store_node(0, tile, sv);
        if (Q == 0 && ntiles == kSegTiles) store_seg(sv);
#pragma unroll
        for (int l = 1; l <= Q; l++) {
            const int span = 1 << l;
            const bool first = (tile & (span - 1)) == 0;
            const bool closes = ((tile + 1) & (span - 1)) == 0;
#pragma unroll
            for (int e = 0; e < DH; e++) acc[l - 1][e] = first ? sv[e] : fmaf(acc[l - 1][e], ge, sv[e]);
            if (closes) {
                const int m = tile >> l;
                if ((m & 1) == 0 && ((m + 1) << l) < NTi) store_node(l, m, acc[l - 1]);
                if (l == Q && ntiles == kSegTiles) store_seg(acc[l - 1]);
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }

    if (!ok || fail_sh) {
        if (tid == 0) record_error(err, kDevTimeout);
        // let in-flight copies and MMAs land before the shared memory and TMEM go away
        for (int b = 0; b < 2; b++) mbar_wait(&bar_mma[b], 0), mbar_wait(&bar_full[b], 0);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kCols);
}

// ------------------------------------------------------------------ tc_merge

// Nodes above the segment level and the per-tile decay table, one launch,
// grid (dk*DV/1024 + 1, max(1, nodes above level q), BH), 256 threads:
//  * block (x >= 1, y): elements [1024 (x-1), 1024 x) of the y-th node (p, m) with
//    p > q that a tile reads (m even, (m+1) 2^p < NT): the decayed sum of its block's
//    full-segment totals (fp32, each decayed to its segment's end),
//    node = sum_sigma exp(log-decay from sigma's end to the block end) Z_sigma.
//    Every input is read independently; no level depends on another.
//  * block (0, 0): the per-tile decay table dtab[bh][j][p] (log2 units): sum of g over
//    tiles [(j >> p) << p, j), the log-decay from the end of node (p, (j >> p) - 1) to
//    the start of tile j, for each set bit p of j.
__global__ void __launch_bounds__(256)
    tc_merge_kernel(const float* __restrict__ seg_tot, const float* __restrict__ g_tiles,
                    __nv_bfloat16* __restrict__ nodes, float* __restrict__ dtab, int* __restrict__ tile_counter,
                    int NT, int q, int P, int nseg, int node_count, int msz, const __grid_constant__ LevelOffsets lo,
                    int T, const SeqMap sm) {
    __shared__ float wsg[1024];      // per-segment totals, then weights, of this block's node
    extern __shared__ float g_sh[];  // the head's tile totals (decay-table block only)
    grid_dep_wait();                 // the node kernel's totals (launched early, see launch_pdl)
    grid_dep_launch();
    const int bh = blockIdx.z;
    const float* gh = g_tiles + static_cast<size_t>(bh) * NT;
    int rowbase, len;
    seq_of(sm, bh, T, rowbase, len);
    const int NTi = (len + kTile - 1) / kTile;  // this head's tiles (NT in the dense layout)
    if (blockIdx.x == 0) {
        if (blockIdx.y != 0) return;
        for (int i = threadIdx.x; i < NTi; i += blockDim.x) g_sh[i] = gh[i];
        __syncthreads();
        for (int j = threadIdx.x; j < NTi; j += blockDim.x) {
            float d[16];
#pragma unroll
            for (int p = 0; p < 16; p++) d[p] = 0.f;
            // walk down from tile j-1, closing the sum at each level's block boundary
            float acc = 0.f;
            int i = j - 1;
#pragma unroll
            for (int p = 0; p < 16; p++) {
                if (p < P && ((j >> p) & 1)) {
                    const int start = (j >> p) << p;
                    for (; i >= start; i--) acc += g_sh[i];
                    d[p] = acc * kLog2e;
                }
            }
            float4* dst = reinterpret_cast<float4*>(dtab + (static_cast<size_t>(bh) * NT + j) * 16);
#pragma unroll
            for (int c = 0; c < 4; c++) dst[c] = make_float4(d[4 * c], d[4 * c + 1], d[4 * c + 2], d[4 * c + 3]);
        }
        return;
    }
    // which node (p, m) is block y
    int y = blockIdx.y, p = q + 1, m = -1;
    for (; p < P; p++) {
        const int cnt = (((NT - 1) >> p) + 1) / 2;
        if (y < cnt) { m = 2 * y; break; }
        y -= cnt;
    }
    if (m < 0 || ((m + 1) << p) >= NTi) return;  // no such node, or no tile of this head reads it
    const int nsg = 1 << (p - q);      // segments in the block
    const int sg0 = m * nsg;           // its first segment
    const int seg_tiles = 1 << q;
    // segment log-decay totals, then each segment's weight exp(sum of the totals after it)
    for (int sg = threadIdx.x; sg < nsg; sg += blockDim.x) {
        float tot = 0.f;
        for (int u = 0; u < seg_tiles; u++) tot += gh[(sg0 + sg) * seg_tiles + u];
        wsg[sg] = tot;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float after = 0.f;
        for (int sg = nsg - 1; sg >= 0; sg--) {
            const float tot = wsg[sg];
            wsg[sg] = expf(after);
            after += tot;
        }
    }
    __syncthreads();
    const int e = (blockIdx.x - 1) * 1024 + threadIdx.x;
    const float* z = seg_tot + (static_cast<size_t>(bh) * nseg + sg0) * msz + e;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int sg = 0; sg < nsg; sg++) {
        const float w = wsg[sg];
#pragma unroll
        for (int i = 0; i < 4; i++) acc[i] = fmaf(w, z[static_cast<size_t>(sg) * msz + 256 * i], acc[i]);
    }
    __nv_bfloat16* dst = nodes + (static_cast<size_t>(bh) * node_count + lo.off[p] + (m >> 1)) * msz + e;
#pragma unroll
    for (int i = 0; i < 4; i++) dst[256 * i] = __float2bfloat16_rn(acc[i]);
}

// ------------------------------------------------------------------ tc_output

// Persistent, warp-specialised output kernel. Each CTA walks tiles
// idx = blockIdx.x + k * gridDim.x (head-major order, so the CTAs running at
// one time share a few heads' nodes in L2). Roles (11 warps):
//   warp 0        input producer: TMA of Q, K, V and bulk copies of the
//                 tile's in-tile decay prefix cl_t (log2 units) and column
//                 weights exp(cl_{s|31} - cl_s) (both written by tc_nodes)
//                 into input stage k % kStages; its 32 lanes add lambda
//                 levels 0..7 of every row with 4-byte cp.async copies.
//   warp 1        MMA issuer (one lane): S_k = Q K^T into TMEM buffer k % 2;
//                 then O = P V and L_p = Q B_p into the O and level slots of
//                 TMEM, kLvSlots levels per round.
//   warp 2        node producer (one lane): the Fenwick nodes each tile reads,
//                 in order, into a ring of shared-memory slots.
//   warps 3-10    epilogue, two warps per TMEM lane quadrant (thread = query
//                 row), each owning half of the columns, with no barrier among
//                 them. Phase 1 builds P_k (bf16, into the K buffer of the
//                 tile's stage) from S_k; phase 2 writes O + sum_p r_p L_p with
//                 r_p = lambda_t^(8+p) exp(cl_t + D_p), whose inputs are fetched
//                 while phase 1 of the next tile runs.
// With two input stages the input producer and the MMA warp run one tile
// ahead (phase 1 of tile k+1 before phase 2 of tile k) and the epilogue
// builds P of tile k+1 before finishing tile k. All hand-offs are mbarriers;
// every wait is bounded.
template <int DV>
struct OutCfg {
    static constexpr int kStages = DV == 64 ? 2 : 1;
    static constexpr int kQ = 0;
    static constexpr int kK = 2 * kPanelBytes;  // K tile, then P of the same tile
    static constexpr int kV = 4 * kPanelBytes;
    static constexpr int kCl2 = kV + (DV / 64) * kPanelBytes;  // 128 floats: in-tile log2 decay prefix
    static constexpr int kScalarTx = 2 * 512;                    // cl2 + colw bulk copies
    static constexpr int kColw = kCl2 + 512;                     // 128 floats: column weights
    static constexpr int kLam8 = kColw + 512;                    // 128 x 8 floats: lambda levels 0..7
    static constexpr int kStageBytes = (kLam8 + kTile * 8 * 4 + 1023) / 1024 * 1024;
    static constexpr int kQkvBytes = (4 + DV / 64) * kPanelBytes;
    static constexpr int kNodeBytes = (DV / 64) * kPanelBytes;
    // TMEM: S of the two tiles in flight at columns [128 b, 128 b + 128). Once a tile's
    // S is consumed its buffer takes the tile's O (first DV columns) and, for DV = 64,
    // level slot 0; the other level slots sit at [256, 512).
    static constexpr int kLvSlots = DV == 64 ? 5 : 2;
    static constexpr int kNodeSlots = DV == 64 ? 3 : 2;
    static constexpr int kNodeBase = kStages * kStageBytes;
    static constexpr int kBytes = kNodeBase + kNodeSlots * kNodeBytes + 1024;
    static constexpr uint32_t kTmemCols = 512;
    __device__ static constexpr uint32_t col_o(int b) { return 128u * b; }
    __device__ static constexpr uint32_t col_lv(int b, int slot) {
        return DV == 64 ? (slot == 0 ? 128u * b + 64u : 256u + 64u * (slot - 1)) : 256u + 128u * slot;
    }
    static constexpr int kEpiWarps = 8;
    static constexpr int kThreads = (3 + kEpiWarps) * 32;
};

// 4-byte asynchronous global -> shared copy (no alignment beyond 4 bytes needed).
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.shared.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <int DV>
__global__ void __launch_bounds__(OutCfg<DV>::kThreads, 1)
    tc_output_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_nodes,
                     const float* __restrict__ tok_cl2, const float* __restrict__ tok_colw,
                     const float* __restrict__ lambda, const float* __restrict__ dtab,
                     __nv_bfloat16* __restrict__ out, int T, int NT, int L, int P, int node_count, const __grid_constant__ LevelOffsets lo,
                     int total_tiles, int* __restrict__ tile_counter, int* err) {
    using C = OutCfg<DV>;
    constexpr int NS = C::kStages;
    constexpr int DH = DV / 2;  // columns of O per epilogue warp
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t in_full[NS], in_empty[NS], s_full[2], s_free[2], p_ready[2];
    __shared__ uint64_t node_full[C::kNodeSlots], node_empty[C::kNodeSlots];
    __shared__ uint64_t lv_full, lv_free, drain, id_ready[NS];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int tile_id_sh[NS];  // tile of the job in each input stage, -1 = no more tiles
    __shared__ volatile int fail_sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < NS; s++) {
            mbar_init(&in_full[s], 2);  // TMA/bulk bytes + lane 0's arrive; the lambda cp.asyncs add their own
            mbar_init(&in_empty[s], 1);
            mbar_init(&id_ready[s], 1);
        }
        for (int s = 0; s < 2; s++) {
            mbar_init(&s_full[s], 1);
            mbar_init(&s_free[s], C::kEpiWarps);
            mbar_init(&p_ready[s], C::kEpiWarps);
        }
        for (int s = 0; s < C::kNodeSlots; s++) {
            mbar_init(&node_full[s], 1);
            mbar_init(&node_empty[s], 1);
        }
        mbar_init(&lv_full, 1);
        mbar_init(&lv_free, C::kEpiWarps);
        mbar_init(&drain, 1);
        fence_mbar_init();
        fail_sh = 0;
    }
    if (warp == 1) tmem_alloc(&tmem_base_sh, C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    grid_dep_wait();  // the node and merge kernels' outputs (launched early, see launch_pdl)

    // Tiles are handed out by a global counter (zeroed by tc_merge), head by head and,
    // within a head, from the last tile down: the tiles with the most Fenwick levels
    // start first and the cheap ones fill the tail.
    auto tile_of = [&](int idx, int& bh, int& j) {
        bh = idx / NT;
        j = NT - 1 - (idx - bh * NT);
    };
    // single-thread bounded wait; after a failure anywhere it returns false at once
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (fail_sh) return false;
        if (mbar_wait(bar, parity)) return true;
        fail_sh = 1;
        record_error(err, kDevTimeout);
        return false;
    };
    // warp-uniform bounded wait with the same failure short-cut
    auto ewait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (__any_sync(0xffffffffu, fail_sh != 0)) return false;
        if (warp_wait(bar, parity)) return true;
        if (lane == 0) {
            fail_sh = 1;
            record_error(err, kDevTimeout);
        }
        return false;
    };

    if (warp == 0) {
        // ---------------------------------------------------------------- input producer
        // Tiles are claimed kClaimAhead jobs before their stage frees up; a claimed
        // tile's Q, K, V, decay rows and lambda rows are pulled into L2 at once, so the
        // stage's own copies later come from L2.
        constexpr int kClaimAhead = 2;
        int claimed[kClaimAhead + 1];
        int n_in = 0;
        auto claim = [&]() -> int {
            int idx = 0;
            if (lane == 0) idx = atomicAdd(tile_counter, 1);
            idx = __shfl_sync(0xffffffffu, idx, 0);
            if (idx >= total_tiles) return -1;
            if (lane == 0) {
                int pbh, pj;
                tile_of(idx, pbh, pj);
                const int r0 = pbh * T + pj * kTile;
                tma_prefetch_l2(&tm_q, 0, r0);
                tma_prefetch_l2(&tm_q, 64, r0);
                tma_prefetch_l2(&tm_k, 0, r0);
                tma_prefetch_l2(&tm_k, 64, r0);
#pragma unroll
                for (int c = 0; c < DV / 64; c++) tma_prefetch_l2(&tm_v, 64 * c, r0);
                prefetch_l2(tok_cl2 + r0, 512);
                prefetch_l2(tok_colw + r0, 512);
                const uintptr_t lb = reinterpret_cast<uintptr_t>(lambda + static_cast<size_t>(r0) * L) & ~uintptr_t(15);
                const uintptr_t le = (reinterpret_cast<uintptr_t>(lambda + static_cast<size_t>(r0 + kTile) * L) + 15) &
                                     ~uintptr_t(15);
                prefetch_l2(reinterpret_cast<const void*>(lb), static_cast<uint32_t>(le - lb));
            }
            return idx;
        };
        for (int a = 0; a < kClaimAhead; a++) claimed[a] = claim();
        for (int k = 0;; k++) {
            const int s = k % NS;
            if (k >= NS && !ewait(&in_empty[s], ((k / NS) - 1) & 1)) break;
            const int idx = claimed[0];
#pragma unroll
            for (int a = 0; a + 1 < kClaimAhead; a++) claimed[a] = claimed[a + 1];
            claimed[kClaimAhead - 1] = idx < 0 ? -1 : claim();
            const bool done = idx < 0;
            if (lane == 0) {
                tile_id_sh[s] = done ? -1 : idx;
                mbar_arrive(&id_ready[s]);
            }
            if (done) {
                if (lane == 0) {
                    mbar_arrive(&in_full[s]);
                    mbar_arrive(&in_full[s]);
                }
                break;
            }
            int bh, j;
            tile_of(idx, bh, j);
            const int row0 = bh * T + j * kTile;
            uint8_t* st = smem + s * C::kStageBytes;
            if (lane == 0) {
                mbar_expect_tx(&in_full[s], C::kQkvBytes + C::kScalarTx);
                tma_load_2d(st + C::kQ, &tm_q, &in_full[s], 0, row0);
                tma_load_2d(st + C::kQ + kPanelBytes, &tm_q, &in_full[s], 64, row0);
                tma_load_2d(st + C::kK, &tm_k, &in_full[s], 0, row0);
                tma_load_2d(st + C::kK + kPanelBytes, &tm_k, &in_full[s], 64, row0);
#pragma unroll
                for (int c = 0; c < DV / 64; c++)
                    tma_load_2d(st + C::kV + c * kPanelBytes, &tm_v, &in_full[s], 64 * c, row0);
                bulk_load(st + C::kCl2, tok_cl2 + row0, 512, &in_full[s]);
                bulk_load(st + C::kColw, tok_colw + row0, 512, &in_full[s]);
            }
            // lambda_t^(0..7) of the tile's 128 rows (rows are L floats apart, not 16-byte aligned);
            // consecutive lanes fill consecutive words of lam8[t][l] (no bank conflicts)
            float* lam8 = reinterpret_cast<float*>(st + C::kLam8);
#pragma unroll 8
            for (int i = 0; i < 32; i++) {
                const int x = lane + 32 * i, t = x >> 3, l = x & 7;
                cp_async4(lam8 + x, lambda + static_cast<size_t>(row0 + t) * L + l);
            }
            cp_async_arrive(&in_full[s]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&in_full[s]);
            n_in = k + 1;
        }
        if (fail_sh && lane == 0) {
            // let this CTA's copies land before its shared memory is released
            for (int k = n_in - NS; k < n_in; k++)
                if (k >= 0) mbar_wait(&in_full[k % NS], (k / NS) & 1);
        }
    } else if (warp == 2) {
        // ---------------------------------------------------------------- node producer
        if (lane == 0) {
            int gn = 0;
            bool ok = true;
            for (int k = 0; ok; k++) {
                if (!wait(&id_ready[k % NS], (k / NS) & 1)) break;
                const int idx = tile_id_sh[k % NS];
                if (idx < 0) break;
                int bh, j;
                tile_of(idx, bh, j);
                for (int p = 0; p < P; p++) {
                    if (((j >> p) & 1) == 0) continue;
                    const int slot = gn % C::kNodeSlots;
                    if (gn >= C::kNodeSlots && !wait(&node_empty[slot], ((gn / C::kNodeSlots) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    const int m = (j >> p) - 1;
                    const int nrow = (bh * node_count + lo.off[p] + (m >> 1)) * kDk;
                    mbar_expect_tx(&node_full[slot], C::kNodeBytes);
#pragma unroll
                    for (int c = 0; c < DV / 64; c++)
                        tma_load_2d(smem + C::kNodeBase + slot * C::kNodeBytes + c * kPanelBytes, &tm_nodes,
                                    &node_full[slot], 64 * c, nrow);
                    gn++;
                }
            }
            if (fail_sh) {
                for (int g = gn - C::kNodeSlots; g < gn; g++)
                    if (g >= 0) mbar_wait(&node_full[g % C::kNodeSlots], (g / C::kNodeSlots) & 1);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int gn = 0, round = 0;
            constexpr uint32_t kIdS = idesc_bf16(kTile, kTile, 0, 0);
            constexpr uint32_t kIdO = idesc_bf16(kTile, DV, 0, 1);
            // phase 1 of the k-th job: returns its tile, -1 when the tiles are exhausted, -2 on failure
            auto phase1 = [&](int k) -> int {
                const int s = k % NS, b = k & 1;
                if (!wait(&in_full[s], (k / NS) & 1)) return -2;
                const int idx = tile_id_sh[s];
                if (idx < 0) return -1;
                if (k >= 2 && !wait(&s_free[b], ((k >> 1) - 1) & 1)) return -2;
                tc_fence_after();
                const uint32_t qb = smem_u32(smem + s * C::kStageBytes + C::kQ);
                const uint32_t kb = smem_u32(smem + s * C::kStageBytes + C::kK);
#pragma unroll
                for (int kk = 0; kk < kDk / 16; kk++) {
                    const uint32_t off = (kk >> 2) * kPanelBytes + (kk & 3) * 32;
                    mma_bf16(tmem + b * kTile, sdesc(qb + off, 16, 1024), sdesc(kb + off, 16, 1024), kIdS,
                             kk > 0 ? 1u : 0u);
                }
                mma_commit(&s_full[b]);
                return idx;
            };
            // Phase 2 of tile k: O = P V into the tile's retired S buffer and the level reads,
            // kLvSlots per round.
            int p2_p = 0, p2_rounds = 0;
            auto phase2 = [&](int k, int idx, bool first_round) -> bool {
                int bh, j;
                tile_of(idx, bh, j);
                const int s = k % NS, b = k & 1;
                if (first_round) {
                    if (!wait(&p_ready[b], (k >> 1) & 1)) return false;
                    tc_fence_after();
                    const int n_lv = __popc(static_cast<unsigned>(j) & ((1u << P) - 1u));
                    p2_rounds = n_lv == 0 ? 1 : (n_lv + C::kLvSlots - 1) / C::kLvSlots;
                    p2_p = 0;
                }
                const uint32_t qb = smem_u32(smem + s * C::kStageBytes + C::kQ);
                const uint32_t pb = smem_u32(smem + s * C::kStageBytes + C::kK);
                const uint32_t vb = smem_u32(smem + s * C::kStageBytes + C::kV);
                const int r_begin = first_round ? 0 : 1;
                const int r_end = first_round ? 1 : p2_rounds;
                for (int r = r_begin; r < r_end; r++, round++) {
                    if (round > 0 && !wait(&lv_free, (round - 1) & 1)) return false;
                    tc_fence_after();
                    if (r == 0) {
#pragma unroll
                        for (int kk = 0; kk < kTile / 16; kk++) {
                            const uint32_t aoff = (kk >> 2) * kPanelBytes + (kk & 3) * 32;
                            mma_bf16(tmem + C::col_o(b), sdesc(pb + aoff, 16, 1024),
                                     sdesc(vb + kk * 2048, kPanelBytes, 1024), kIdO, kk > 0 ? 1u : 0u);
                        }
                    }
                    for (int sl = 0; sl < C::kLvSlots; sl++) {
                        while (p2_p < P && ((j >> p2_p) & 1) == 0) p2_p++;
                        if (p2_p >= P) break;
                        p2_p++;
                        const int slot = gn % C::kNodeSlots;
                        // Two levels in one MMA chain (N = 128, Q read once) when the next level's
                        // node sits in the next ring slot (16 KB further: the B operand's panel
                        // stride) and its TMEM level slot follows this one (slots 1.. are contiguous).
                        int p_next = p2_p;
                        while (p_next < P && ((j >> p_next) & 1) == 0) p_next++;
                        const bool pair = DV == 64 && sl >= 1 && sl + 1 < C::kLvSlots && p_next < P &&
                                          slot + 1 < C::kNodeSlots;
                        if (!wait(&node_full[slot], (gn / C::kNodeSlots) & 1)) return false;
                        if (pair && !wait(&node_full[slot + 1], ((gn + 1) / C::kNodeSlots) & 1)) return false;
                        tc_fence_after();
                        const uint32_t nb = smem_u32(smem + C::kNodeBase + slot * C::kNodeBytes);
                        const uint32_t dcol = C::col_lv(b, sl);
                        if (pair) {
                            constexpr uint32_t kIdO2 = idesc_bf16(kTile, 2 * DV, 0, 1);
#pragma unroll
                            for (int kk = 0; kk < kDk / 16; kk++) {
                                const uint32_t aoff = (kk >> 2) * kPanelBytes + (kk & 3) * 32;
                                mma_bf16(tmem + dcol, sdesc(qb + aoff, 16, 1024),
                                         sdesc(nb + kk * 2048, kPanelBytes, 1024), kIdO2, kk > 0 ? 1u : 0u);
                            }
                            mma_commit(&node_empty[slot]);
                            mma_commit(&node_empty[slot + 1]);
                            gn += 2;
                            p2_p = p_next + 1;
                            sl++;
                            continue;
                        }
#pragma unroll
                        for (int kk = 0; kk < kDk / 16; kk++) {
                            const uint32_t aoff = (kk >> 2) * kPanelBytes + (kk & 3) * 32;
                            mma_bf16(tmem + dcol, sdesc(qb + aoff, 16, 1024), sdesc(nb + kk * 2048, kPanelBytes, 1024),
                                     kIdO, kk > 0 ? 1u : 0u);
                        }
                        mma_commit(&node_empty[slot]);
                        gn++;
                    }
                    mma_commit(&lv_full);
                }
                if (r_end == p2_rounds) mma_commit(&in_empty[s]);  // every MMA of the tile is issued
                return true;
            };
            // Order: phase 1 of tile 0; then per tile k: phase 2 of k (all rounds), phase 1
            // of k+1. The next tile's S is computed while the epilogue finishes tile k.
            int id_cur = phase1(0);
            for (int k = 0; id_cur >= 0; k++) {
                if (!phase2(k, id_cur, true)) break;
                if (p2_rounds > 1 && !phase2(k, id_cur, false)) break;
                id_cur = phase1(k + 1);
            }
            // every MMA issued by this CTA has completed before TMEM is released
            mma_commit(&drain);
            mbar_wait(&drain, 0);
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int ew = warp - 3;
        const int quad = warp & 3;
        const int half = ew >> 2;
        (void)quad;
        const int t = quad * 32 + lane;  // query row of the tile = TMEM lane
        const int q32 = quad * 32;
        const uint32_t lane_base = static_cast<uint32_t>(q32) << 16;
        int round = 0;

        // Inputs of phase 2 of a tile, fetched one phase early: lambda_t^(8+p) and the
        // decay-table row of the tile, plus the row's decay prefix.
        float pre_lam[16], pre_d[16];
        float cl2_even = 0.f, cl2_odd = 0.f;
        auto prefetch2 = [&](int idx) {
            int bh, j;
            tile_of(idx, bh, j);
            const int row0 = bh * T + j * kTile;
            const float* lam_row = lambda + static_cast<size_t>(row0 + t) * L;
            const float4* drow = reinterpret_cast<const float4*>(dtab + (static_cast<size_t>(bh) * NT + j) * 16);
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const float4 x = drow[c];
                pre_d[4 * c] = x.x; pre_d[4 * c + 1] = x.y; pre_d[4 * c + 2] = x.z; pre_d[4 * c + 3] = x.w;
            }
#pragma unroll
            for (int p = 0; p < 16; p++) pre_lam[p] = (p < P && ((j >> p) & 1)) ? lam_row[8 + p] : 0.f;
        };

        // Phase 1: P_k. The two warps of a lane quadrant split every 32-key chunk,
        // 16 keys each, so the masked diagonal chunk is shared evenly.
        // returns the job's tile, -1 at the end marker or on failure
        auto epi1 = [&](int k) -> int {
            const int s = k % NS, b = k & 1;
            const uint8_t* st = smem + s * C::kStageBytes;
            if (!ewait(&in_full[s], (k / NS) & 1)) return -1;
            const int idx = tile_id_sh[s];
            if (idx < 0) return -1;
            const float* cl2 = reinterpret_cast<const float*>(st + C::kCl2);
            const float* colw = reinterpret_cast<const float*>(st + C::kColw);
            const float cl2_t = cl2[t];
            if (b) cl2_odd = cl2_t; else cl2_even = cl2_t;
            float lam_in[8];
            const float4* lam8 = reinterpret_cast<const float4*>(st + C::kLam8) + t * 2;
            {
                const float4 x0 = lam8[0], x1 = lam8[1];
                lam_in[0] = x0.x; lam_in[1] = x0.y; lam_in[2] = x0.z; lam_in[3] = x0.w;
                lam_in[4] = x1.x; lam_in[5] = x1.y; lam_in[6] = x1.z; lam_in[7] = x1.w;
            }
            if (!ewait(&s_full[b], (k >> 1) & 1)) return -1;
            tc_fence_after();
            uint8_t* pbase = smem + s * C::kStageBytes + C::kK;
#pragma unroll 1
            for (int c0 = 0; c0 < kTile; c0 += 32) {
                const int cb = c0 + half * 16;  // first key of this warp's 16
                uint32_t pk[8];
                if (c0 > q32) {
                    // keys after every query row of this warp
#pragma unroll
                    for (int e = 0; e < 8; e++) pk[e] = 0u;
                } else {
                    float sv[16];
                    tmem_ld16(tmem + lane_base + b * kTile + cb, sv);
                    if (c0 < q32) {
                        // keys before every row of this warp: one level per row, factorised decay
                        const int lvl = 32 - __clz(t ^ c0);
                        float lw = lam_in[0];
#pragma unroll
                        for (int l = 1; l < 8; l++) lw = (lvl == l) ? lam_in[l] : lw;
                        const float rowf = exp2f(cl2_t - cl2[c0 + 31]) * lw;
#pragma unroll
                        for (int e = 0; e < 16; e += 2)
                            pk[e >> 1] = pack_bf16(sv[e] * rowf * colw[cb + e], sv[e + 1] * rowf * colw[cb + e + 1]);
                    } else {
                        // diagonal chunk: causal mask and per-key levels 0..5, branch-free
                        float v[16];
#pragma unroll
                        for (int e = 0; e < 16; e++) {
                            const int sidx = cb + e;
                            const int lvl = 32 - __clz(t ^ sidx);
                            float lw = lam_in[0];
#pragma unroll
                            for (int l = 1; l < 6; l++) lw = (lvl == l) ? lam_in[l] : lw;
                            const float x = sv[e] * exp2f(fminf(cl2_t - cl2[sidx], 0.f)) * lw;
                            v[e] = sidx <= t ? x : 0.f;
                        }
#pragma unroll
                        for (int e = 0; e < 16; e += 2) pk[e >> 1] = pack_bf16(v[e], v[e + 1]);
                    }
                }
                uint8_t* panel = pbase + (c0 >> 6) * kPanelBytes;
                const int chunk0 = (cb & 63) >> 3;
                *reinterpret_cast<uint4*>(panel + sw128_off(t, chunk0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *reinterpret_cast<uint4*>(panel + sw128_off(t, chunk0 + 1)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_ready[b]);
            return idx;
        };

        // Phase 2: O + sum_p r_p L_p for this warp's half of the columns.
        auto epi2 = [&](int k, int idx) {
            int bh, j;
            tile_of(idx, bh, j);
            const int b = k & 1;
            const int row0 = bh * T + j * kTile;
            const float cl2_t = b ? cl2_odd : cl2_even;
            // level weights of the tile's set bits, in level order
            float rr[16];
            int nl = 0;
#pragma unroll
            for (int p = 0; p < 16; p++) {
                const float w = pre_lam[p] * exp2f(cl2_t + pre_d[p]);
                if (p < P && ((j >> p) & 1)) rr[nl++] = w;
            }
            float acc[DH];
            const int rounds = nl == 0 ? 1 : (nl + C::kLvSlots - 1) / C::kLvSlots;
            for (int r = 0; r < rounds; r++, round++) {
                if (!ewait(&lv_full, round & 1)) return;
                tc_fence_after();
                if (r == 0) {
#pragma unroll
                    for (int c0 = 0; c0 < DH; c0 += 32) tmem_ld32(tmem + lane_base + C::col_o(b) + half * DH + c0, acc + c0);
                }
                const int x_end = min(nl, (r + 1) * C::kLvSlots);
#pragma unroll 1
                for (int x = r * C::kLvSlots; x < x_end; x++) {
                    const float w = rr[x];
                    const uint32_t col = C::col_lv(b, x - r * C::kLvSlots) + half * DH;
#pragma unroll
                    for (int c0 = 0; c0 < DH; c0 += 32) {
                        float lvv[32];
                        tmem_ld32(tmem + lane_base + col + c0, lvv);
#pragma unroll
                        for (int e = 0; e < 32; e++) acc[c0 + e] = fmaf(w, lvv[e], acc[c0 + e]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&lv_free);
            }
            // the tile's TMEM buffer may now take the S of the tile two jobs ahead
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[b]);
            // whole 64-byte runs of 8 rows per warp store (rows q32 + (lane & ~3) + i)
#pragma unroll
            for (int cb = 0; cb < DH / 32; cb++) {
                uint4 x[4];
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    const float* a = acc + 32 * cb + 8 * c;
                    x[c] = make_uint4(pack_bf16(a[0], a[1]), pack_bf16(a[2], a[3]), pack_bf16(a[4], a[5]),
                                      pack_bf16(a[6], a[7]));
                }
                lane_group_transpose(x, lane);
#pragma unroll
                for (int i = 0; i < 4; i++)
                    *reinterpret_cast<uint4*>(out + static_cast<size_t>(row0 + q32 + (lane & ~3) + i) * DV + half * DH +
                                              32 * cb + 8 * (lane & 3)) = x[i];
            }
        };

        for (int k = 0;; k++) {
            const int id = epi1(k);
            if (id < 0) break;
            prefetch2(id);
            epi2(k, id);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

// ------------------------------------------------------------------ tc_output_pp (dv = 64)

// Weights of the 16 keys s = 32 blk + 16 half + e (e = 0..15) of a diagonal 32 x 32 block for the
// query in lane `lane` of the block: lx[l] for the level l = 1 + floor(log2(lane ^ s')) of the
// pair (lx[0] at s' = lane; s' = s mod 32), 0 where s' > lane (the highest differing bit is set in
// s'), times the key's column weight cw[e]. Bits 0..3 of s' are e, fixed at compile time, so each
// of their tests is a per-lane predicate; bit 4 (the half) is decided once per lane.
__device__ __forceinline__ void diag_weights(int lane, int half, const float* lx, const float* cw, float* w) {
    bool lb[4];
#pragma unroll
    for (int b = 0; b < 4; b++) lb[b] = (lane >> b) & 1;
    const bool diff4 = ((lane >> 4) & 1) != half;  // the key is in the other 16-key half
    const float v4 = half ? 0.f : lx[5];           // key after every such row, or before it
    const float4* cw4 = reinterpret_cast<const float4*>(cw);
    float c[16];
#pragma unroll
    for (int e4 = 0; e4 < 4; e4++) {
        const float4 x = cw4[e4];
        c[4 * e4] = x.x; c[4 * e4 + 1] = x.y; c[4 * e4 + 2] = x.z; c[4 * e4 + 3] = x.w;
    }
#pragma unroll
    for (int e = 0; e < 16; e++) {
        float v = lx[0];
#pragma unroll
        for (int b = 0; b < 4; b++) {
            const bool sb = (e >> b) & 1;
            v = (lb[b] != sb) ? (sb ? 0.f : lx[b + 1]) : v;  // higher bits override lower ones
        }
        v = diff4 ? v4 : v;
        w[e] = v * c[e];
    }
}

// Ping-pong output kernel for dv = 64: two independent tile pipelines share one CTA.
// Epilogue group g (eight warps, two per TMEM lane quadrant; thread = query row)
// owns input stage g and TMEM columns [256 g, 256 g + 256) and takes every other
// tile the CTA claims, so one group builds its tile's P while the other group's
// level and PV products run on the tensor pipe. Roles (20 warps):
//   warps 0, 1  producers of groups 0 and 1 (one lane each): claim the group's next
//               tile from the dynamic counter and pull it into L2; once the group's
//               stage is free, TMA of Q, K, V and a bulk copy of the tile's column
//               decay weights into it, then the Fenwick nodes the tile reads, in level
//               order, into the group's two-slot node ring.
//   warps 2, 3  MMA issuers of groups 0 and 1 (one lane each).
//   warps 4-11  epilogue of group 0; warps 12-19 epilogue of group 1. The two warps
//               of a lane quadrant split every 32-key block of P (16 keys each) and
//               the dv columns of the result (32 each).
// TMEM of a group, per tile:
//   round 0: S = Q K^T in [0, 128); the first two level reads L_p = Q B_p in
//            [128, 192) and [192, 256) (they overlap the build of P);
//   round 1: O = P V in [0, 64) once P is in shared memory (over K), and up to
//            three more level reads in [64, 128), [128, 192), [192, 256);
//   round r >= 2: three more level reads each in [64, 256).
// The epilogue reads every round back into fp32 accumulators,
// acc = O + sum_p lambda_t^(8+p) exp(cl_t + D_p) L_p, and stores them as bf16 (whole
// 64-byte runs of rows, through the lane-group transpose).
struct PpCfg {
    static constexpr int kQ = 0;
    static constexpr int kK = 2 * kPanelBytes;  // K tile, then P of the same tile
    static constexpr int kV = 4 * kPanelBytes;
    static constexpr int kQkvBytes = 5 * kPanelBytes;
    static constexpr int kStageBytes = kQkvBytes;
    static constexpr int kNodeSlots = 2;  // per group
    static constexpr int kNodeBytes = kPanelBytes;
    static constexpr int kNodeBase = 2 * kStageBytes;
    // 128 floats per group after the node slots: the tile's column decay weights
    // 2^(cl_{s|31} - cl_s) (key s to the end of its 32-key block)
    static constexpr int kColwBase = kNodeBase + 2 * kNodeSlots * kNodeBytes;
    static constexpr int kScalarTx = 512;
    static constexpr int kBytes = kColwBase + 2 * 512 + 1024;
    static constexpr int kEpiWarps = 8;  // per group
    static constexpr int kFirstEpi = 4;  // first epilogue warp
    static constexpr int kThreads = (kFirstEpi + 2 * kEpiWarps) * 32;
    static constexpr int kR0 = 2;  // level reads in round 0
    static constexpr int kRn = 3;  // level reads in each later round
    __host__ __device__ static constexpr int rounds(int n_lv) {
        return n_lv <= kR0 + kRn ? 2 : 2 + (n_lv - kR0 - kRn + kRn - 1) / kRn;
    }
    // first level (index into the tile's list of set bits) of round r, and the TMEM column of its i-th read
    __host__ __device__ static constexpr int round_begin(int r) { return r == 0 ? 0 : kR0 + (r - 1) * kRn; }
    __host__ __device__ static constexpr int round_size(int r) { return r == 0 ? kR0 : kRn; }
    __device__ static constexpr uint32_t lv_col(int r, int i) { return r == 0 ? 128u + 64u * i : 64u + 64u * i; }
};
static_assert(PpCfg::kBytes <= 232448 - 512, "ping-pong output kernel exceeds shared memory");

__global__ void __launch_bounds__(PpCfg::kThreads, 1)
    tc_output_pp_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_nodes,
                        const float* __restrict__ tok_cl2, const float* __restrict__ tok_colw,
                        const float* __restrict__ lambda, const float* __restrict__ dtab,
                        __nv_bfloat16* __restrict__ out, int T, int NT, int L, int P, int node_count,
                        const __grid_constant__ LevelOffsets lo, int total_tiles, int* __restrict__ tile_counter,
                        const SeqMap sm, int in_rows, int* err) {
    constexpr int DV = 64;
    constexpr int DH = DV / 2;  // result columns per epilogue warp
    using C = PpCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t in_full[2], in_empty[2], kv_empty[2], s_full[2], p_ready[2], lv_full[2], lv_free[2], drain[2];
    __shared__ uint64_t node_full[2][C::kNodeSlots], node_empty[2][C::kNodeSlots];
    __shared__ uint64_t never;  // nothing arrives at it (failure-path test hook)
    __shared__ uint32_t tmem_base_sh;
    __shared__ int tile_id_sh[2];  // tile of the job in each stage, -1 = no more tiles
    __shared__ volatile int fail_sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int g = 0; g < 2; g++) {
            mbar_init(&in_full[g], 1);  // the producer's expect_tx arrive + the bytes
            mbar_init(&in_empty[g], 1);
            mbar_init(&kv_empty[g], 1);
            mbar_init(&s_full[g], 1);
            mbar_init(&p_ready[g], C::kEpiWarps);
            mbar_init(&lv_full[g], 1);
            mbar_init(&lv_free[g], C::kEpiWarps);
            mbar_init(&drain[g], 1);
        }
        for (int g = 0; g < 2; g++)
            for (int s = 0; s < C::kNodeSlots; s++) {
                mbar_init(&node_full[g][s], 1);
                mbar_init(&node_empty[g][s], 1);
            }
        mbar_init(&never, 1);
        fence_mbar_init();
        fail_sh = 0;
    }
    if (warp == 2) tmem_alloc(&tmem_base_sh, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    // The node kernel's outputs (decay tables, level 0..q nodes, the tile counter's reset) are
    // complete when this grid starts. The merge kernel's (nodes above level q, the level decay
    // table) are waited for where they are first read: by a producer before its first node copy,
    // by an epilogue thread before its first read-back; the first tiles' Q, K, V copies, S and P
    // run while the merge kernel drains.

    // head-major; within a head from the last tile down (most Fenwick levels first). Packed
    // sequences: sequence-major, then head; the sequence is found in the tile prefix.
    if (sm.seq) total_tiles = sm.tile_prefix[sm.n_seq];
    auto tile_of = [&](int idx, int& bh, int& j) {
        if (!sm.seq) {
            bh = idx / NT;
            j = NT - 1 - (idx - bh * NT);
            return;
        }
        int lo_ = 0, hi_ = sm.n_seq - 1;  // the sequence i with prefix[i] <= idx < prefix[i + 1]
        while (lo_ < hi_) {
            const int mid = (lo_ + hi_ + 1) >> 1;
            if (sm.tile_prefix[mid] <= idx) lo_ = mid; else hi_ = mid - 1;
        }
        const int p0 = sm.tile_prefix[lo_];
        const int nti = (sm.tile_prefix[lo_ + 1] - p0) / sm.H;
        const int r = idx - p0, h = r / nti;
        bh = lo_ * sm.H + h;
        j = nti - 1 - (r - h * nti);
    };
    const long long lim = tc_pipe_wait_limit;
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (fail_sh) return false;
        if (mbar_wait(bar, parity, lim)) return true;
        fail_sh = 1;
        record_error(err, kDevTimeout);
        return false;
    };
    auto ewait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (__any_sync(0xffffffffu, fail_sh != 0)) return false;
        if (warp_wait(bar, parity, lim)) return true;
        if (lane == 0) {
            fail_sh = 1;
            record_error(err, kDevTimeout);
        }
        return false;
    };

    if (warp < 2) {
        // ---------------------------------------------------------------- producer of group g
        const int g = warp;
        if (lane == 0) {
            // a claimed tile's inputs are pulled into L2 at once; the stage copies come later
            auto claimed = [&](int idx) -> int {
                if (idx >= total_tiles) return -1;
                int pbh, pj, prb, plen;
                tile_of(idx, pbh, pj);
                seq_of(sm, pbh, T, prb, plen);
                const int r0 = prb + pj * kTile;
                tma_prefetch_l2(&tm_q, 0, r0);
                tma_prefetch_l2(&tm_q, 64, r0);
                tma_prefetch_l2(&tm_k, 0, r0);
                tma_prefetch_l2(&tm_k, 64, r0);
                tma_prefetch_l2(&tm_v, 0, r0);
                prefetch_l2(tok_cl2 + pbh * T + pj * kTile, 512);
                prefetch_l2(tok_colw + pbh * T + pj * kTile, 512);
                // this tile's lambda rows, within the tensor (a packed tile may end past it)
                const int r1 = min(r0 + kTile, in_rows);
                const uintptr_t lb = reinterpret_cast<uintptr_t>(lambda + static_cast<size_t>(r0) * L) & ~uintptr_t(15);
                const uintptr_t le = reinterpret_cast<uintptr_t>(lambda + static_cast<size_t>(r1) * L) & ~uintptr_t(15);
                if (le > lb) prefetch_l2(reinterpret_cast<const void*>(lb), static_cast<uint32_t>(le - lb));
                return idx;
            };
            uint8_t* st = smem + g * C::kStageBytes;
            uint8_t* ring = smem + C::kNodeBase + g * C::kNodeSlots * C::kNodeBytes;
            int next = claimed(atomicAdd(tile_counter, 1));
            int gn = 0, n_in = 0;
            for (int c = 0;; c++) {
                // K (P) and V of the previous tile are free once PV has read them; Q and the
                // decay prefix once its last level read has
                if (c > 0 && !wait(&kv_empty[g], (c - 1) & 1)) break;
                const int idx = next;
                tile_id_sh[g] = idx;
                if (idx < 0) {
                    mbar_arrive(&in_full[g]);  // end marker
                    break;
                }
                int bh, j, rb, len;
                tile_of(idx, bh, j);
                seq_of(sm, bh, T, rb, len);
                const int row0 = rb + j * kTile;  // input rows
                mbar_expect_tx(&in_full[g], C::kQkvBytes + C::kScalarTx);
                tma_load_2d(st + C::kK, &tm_k, &in_full[g], 0, row0);
                tma_load_2d(st + C::kK + kPanelBytes, &tm_k, &in_full[g], 64, row0);
                tma_load_2d(st + C::kV, &tm_v, &in_full[g], 0, row0);
                n_in = c + 1;
                // (on a failed wait the rest is still copied, so that the phase completes and the
                // clean-up below can wait for every copy of it to land)
                const bool q_free = c == 0 || wait(&in_empty[g], (c - 1) & 1);
                tma_load_2d(st + C::kQ, &tm_q, &in_full[g], 0, row0);
                tma_load_2d(st + C::kQ + kPanelBytes, &tm_q, &in_full[g], 64, row0);
                bulk_load(smem + C::kColwBase + g * 512, tok_colw + bh * T + j * kTile, 512, &in_full[g]);
                if (!q_free) break;
                if (c == 0) grid_dep_wait();  // the merge kernel's nodes
                // claim the group's next tile; its index is used once this tile's node copies are issued
                const int next_idx = atomicAdd(tile_counter, 1);
                // the tile's Fenwick nodes, in level order, into the group's ring
                bool ok = true;
                for (int p = 0; p < P && ok; p++) {
                    if (((j >> p) & 1) == 0) continue;
                    const int slot = gn % C::kNodeSlots;
                    if (gn >= C::kNodeSlots && !wait(&node_empty[g][slot], ((gn / C::kNodeSlots) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    const int m = (j >> p) - 1;
                    const int nrow = (bh * node_count + lo.off[p] + (m >> 1)) * kDk;
                    mbar_expect_tx(&node_full[g][slot], C::kNodeBytes);
                    tma_load_2d(ring + slot * C::kNodeBytes, &tm_nodes, &node_full[g][slot], 0, nrow);
                    gn++;
                }
                if (!ok) break;
                next = claimed(next_idx);
            }
            if (fail_sh) {
                // let this group's copies land before the shared memory is released
                if (n_in > 0) mbar_wait(&in_full[g], (n_in - 1) & 1);
                for (int x = gn - C::kNodeSlots; x < gn; x++)
                    if (x >= 0) mbar_wait(&node_full[g][x % C::kNodeSlots], (x / C::kNodeSlots) & 1);
            }
        }
    } else if (warp < 4) {
        // ---------------------------------------------------------------- MMA issuer of group g
        const int g = warp - 2;
        if (lane == 0) {
            const uint32_t tb = tmem + 256u * g;
            constexpr uint32_t kIdS = idesc_bf16(kTile, kTile, 0, 0);
            constexpr uint32_t kIdO = idesc_bf16(kTile, DV, 0, 1);
            const uint32_t st = smem_u32(smem + g * C::kStageBytes);
            const uint32_t qb = st + C::kQ, kb = st + C::kK, vb = st + C::kV;
            int lvf = 0;  // lv_free phases of this group waited so far
            int gn = 0;   // nodes of this group's ring consumed so far
            const uint32_t ring = smem_u32(smem + C::kNodeBase + g * C::kNodeSlots * C::kNodeBytes);
            // level reads [x0, x1) of the tile, into round r's slots
            auto levels = [&](int x0, int x1, int r) -> bool {
                for (int x = x0; x < x1; x++) {
                    const int slot = gn % C::kNodeSlots;
                    if (!wait(&node_full[g][slot], (gn / C::kNodeSlots) & 1)) return false;
                    tc_fence_after();
                    const uint32_t nb = ring + slot * C::kNodeBytes;
                    const uint32_t dcol = tb + C::lv_col(r, x - x0);
#pragma unroll
                    for (int kk = 0; kk < kDk / 16; kk++) {
                        const uint32_t aoff = (kk >> 2) * kPanelBytes + (kk & 3) * 32;
                        mma_bf16(dcol, sdesc(qb + aoff, 16, 1024), sdesc(nb + kk * 2048, kPanelBytes, 1024), kIdO,
                                 kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&node_empty[g][slot]);
                    gn++;
                }
                return true;
            };
            for (int c = 0;; c++) {
                if (!wait(&in_full[g], c & 1)) break;
                const int idx = tile_id_sh[g];
                if (idx < 0) break;
                int tbh, tj;
                tile_of(idx, tbh, tj);
                const int n_lv = __popc(static_cast<unsigned>(tj));
                const int R = C::rounds(n_lv);
                // the previous tile of this group is read back: its TMEM columns are free
                if (c > 0 && !wait(&lv_free[g], (lvf++) & 1)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kDk / 16; kk++) {
                    const uint32_t off = (kk >> 2) * kPanelBytes + (kk & 3) * 32;
                    mma_bf16(tb, sdesc(qb + off, 16, 1024), sdesc(kb + off, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
                }
                mma_commit(&s_full[g]);
                bool ok = levels(0, min(n_lv, C::kR0), 0);
                if (!ok) break;
                mma_commit(&lv_full[g]);
                // round 1: O = P V once P has replaced K, then the next level reads
                if (!wait(&p_ready[g], c & 1)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kTile / 16; kk++) {
                    const uint32_t aoff = (kk >> 2) * kPanelBytes + (kk & 3) * 32;
                    mma_bf16(tb, sdesc(kb + aoff, 16, 1024), sdesc(vb + kk * 2048, kPanelBytes, 1024), kIdO,
                             kk > 0 ? 1u : 0u);
                }
                mma_commit(&kv_empty[g]);  // PV has been issued: K (P) and V are read once it completes
                for (int r = 1; r < R && ok; r++) {
                    if (!wait(&lv_free[g], (lvf++) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int x0 = C::round_begin(r);
                    ok = levels(min(n_lv, x0), min(n_lv, x0 + C::round_size(r)), r);
                    if (ok) mma_commit(&lv_full[g]);
                }
                if (!ok) break;
                mma_commit(&in_empty[g]);  // every MMA reading this stage has been issued
            }
            mma_commit(&drain[g]);
            mbar_wait(&drain[g], 0);
        }
    } else {
        // ---------------------------------------------------------------- epilogue of group g
        const int ew = warp - C::kFirstEpi;
        const int g = ew >> 3;
        const int half = (ew >> 2) & 1;
        const int quad = warp & 3;
        const int t = quad * 32 + lane;  // query row = TMEM lane
        const int q32 = quad * 32;
        const uint32_t tb = tmem + 256u * g + (static_cast<uint32_t>(q32) << 16);
        const float* colw = reinterpret_cast<const float*>(smem + C::kColwBase + g * 512);
        int rnd = 0;  // lv_full phases of this group consumed so far
        // test hook: a wait that runs out (records the timeout; every role then leaves)
        const bool held = tc_debug_hold != 0 && !ewait(&never, 0);
        for (int c = 0; !held; c++) {
            if (!ewait(&in_full[g], c & 1)) break;
            const int idx = tile_id_sh[g];
            if (idx < 0) break;
            int bh, j, rb, len;
            tile_of(idx, bh, j);
            seq_of(sm, bh, T, rb, len);
            const int row0 = rb + j * kTile;         // input rows
            const int live = len - j * kTile;        // rows of this tile inside the sequence (>= 1)
            const int tr = t < live ? t : live - 1;  // lambda row read for this lane
            // in-tile log2 decay prefix: this row's and the last of each 32-key block
            const float* cl2 = tok_cl2 + bh * T + j * kTile;
            const float cl2_t = cl2[t];
            float cend[4];
#pragma unroll
            for (int b = 0; b < 4; b++) cend[b] = cl2[32 * b + 31];
            // this row's lambda for levels 0..7 (the weights of P), loaded while S is computed;
            // the rest of the row (levels 8 + p, the weights of the level reads) and the tile's
            // decay-table row are pulled into L1 for the read-back
            float lam_in[8];
            const float* lam_row = lambda + static_cast<size_t>(row0 + tr) * L;
            const float* drow = dtab + (static_cast<size_t>(bh) * NT + j) * 16;
#pragma unroll
            for (int l = 0; l < 8; l++) lam_in[l] = l < L ? lam_row[l] : 0.f;
            if (L > 8) prefetch_l1(lam_row + L - 1);
            if (lane == 0) prefetch_l1(drow);
            // ---- P = (S masked, decayed, lambda-weighted) -> bf16 over K in shared memory
            if (!ewait(&s_full[g], c & 1)) break;
            tc_fence_after();
            uint8_t* pbase = smem + g * C::kStageBytes + C::kK;
            // key chunk ci (32 keys, this warp's 16 of them) is live for the warp's rows when 32 ci <= q32
#pragma unroll 1
            for (int ci = 0; ci < kTile / 32; ci++) {
                const int c0 = ci * 32;
                const int cb = c0 + half * 16;  // first key of this warp's 16
                // the block's last log decay, by selects (an indexed register array would be
                // placed in local memory)
                const float cen = ci == 0 ? cend[0] : ci == 1 ? cend[1] : ci == 2 ? cend[2] : cend[3];
                uint32_t sv[16];
                uint32_t pk[8];
                if (c0 > q32) {
#pragma unroll
                    for (int e = 0; e < 8; e++) pk[e] = 0u;
                } else if (c0 < q32) {
                    // keys before every row of this warp: one level per row (7 if bit 6 of t ^ s
                    // is set, else 6) and the decay factorised at the block end,
                    // 2^(cl_t - cl_s) = 2^(cl_t - cl_{c0+31}) * 2^(cl_{c0+31} - cl_s), both <= 1
                    // for non-positive log decays; the weights are formed while S is loaded
                    const float rowf = ex2_ftz(cl2_t - cen) * (((t ^ c0) & 64) ? lam_in[7] : lam_in[6]);
                    tmem_ld16_issue(tb + cb, sv);
                    float w[16];
                    const float4* cw4 = reinterpret_cast<const float4*>(colw + cb);
#pragma unroll
                    for (int e4 = 0; e4 < 4; e4++) {
                        const float4 x = cw4[e4];
                        w[4 * e4] = rowf * x.x; w[4 * e4 + 1] = rowf * x.y;
                        w[4 * e4 + 2] = rowf * x.z; w[4 * e4 + 3] = rowf * x.w;
                    }
                    tmem_ld16_wait(sv);
#pragma unroll
                    for (int e = 0; e < 16; e += 2)
                        pk[e >> 1] = pack_bf16(__uint_as_float(sv[e]) * w[e], __uint_as_float(sv[e + 1]) * w[e + 1]);
                } else {
                    // diagonal block: the causal mask and a per-key level 1 + floor(log2(t ^ s))
                    // (0 at s = t). Where every column weight of the block lies in [2^-100, 2^100]
                    // the decay is factorised at the block end as above (the row factor is then at
                    // most 2^100, the product exact to a few ulp); else each key's factor is exact.
                    const bool fact = __all_sync(0xffffffffu, colw[c0 + lane] >= 0x1p-100f && colw[c0 + lane] <= 0x1p100f);
                    tmem_ld16_issue(tb + cb, sv);
                    float w[16];
                    if (fact) {
                        const float rowf = ex2_ftz(cl2_t - cen);
                        float lx[6];
#pragma unroll
                        for (int l = 0; l < 6; l++) lx[l] = lam_in[l] * rowf;
                        diag_weights(lane, half, lx, colw + cb, w);
                    } else {
                        // a masked key (s > t) may give an infinite factor; the select drops it
#pragma unroll
                        for (int e = 0; e < 16; e++) {
                            const int sidx = cb + e;
                            const int x = t ^ sidx;
                            float lw = x >= 16 ? lam_in[5] : lam_in[4];
                            lw = x < 8 ? lam_in[3] : lw;
                            lw = x < 4 ? lam_in[2] : lw;
                            lw = x < 2 ? lam_in[1] : lw;
                            lw = x == 0 ? lam_in[0] : lw;
                            w[e] = sidx <= t ? ex2_ftz(cl2_t - cl2[sidx]) * lw : 0.f;
                        }
                    }
                    tmem_ld16_wait(sv);
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        // 0 * S, not a select: S is finite
                        pk[e >> 1] = pack_bf16(__uint_as_float(sv[e]) * w[e], __uint_as_float(sv[e + 1]) * w[e + 1]);
                    }
                }
                uint8_t* panel = pbase + (c0 >> 6) * kPanelBytes;
                const int chunk0 = (cb & 63) >> 3;
                *reinterpret_cast<uint4*>(panel + sw128_off(t, chunk0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *reinterpret_cast<uint4*>(panel + sw128_off(t, chunk0 + 1)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_ready[g]);

            if (c == 0) grid_dep_wait();  // the merge kernel's level decay table
            // ---- read back every round: acc = O + sum_p r_p L_p (this warp's half of the columns)
            const int n_lv = __popc(static_cast<unsigned>(j));
            const int R = C::rounds(n_lv);
            float acc[DH];
#pragma unroll
            for (int e = 0; e < DH; e++) acc[e] = 0.f;
            bool ok = true;
            int p_cur = 0;  // level of the next read
            for (int r = 0; r < R; r++) {
                if (!ewait(&lv_full[g], (rnd++) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (r == 1) {
                    float o[DH];
                    tmem_ld32(tb + half * DH, o);
#pragma unroll
                    for (int e = 0; e < DH; e++) acc[e] += o[e];
                }
                const int x0 = min(n_lv, C::round_begin(r)), x1 = min(n_lv, C::round_begin(r) + C::round_size(r));
#pragma unroll 1
                for (int x = x0; x < x1; x++) {
                    while (((j >> p_cur) & 1) == 0) p_cur++;
                    // lambda_t^(8+p) exp(cl_t + D_p), read where it is used (the row and the
                    // decay-table row are in L1 from the tile's start)
                    const float w = lam_row[8 + p_cur] * exp2f(cl2_t + drow[p_cur]);
                    p_cur++;
                    float lv[DH];
                    tmem_ld32(tb + C::lv_col(r, x - x0) + half * DH, lv);
#pragma unroll
                    for (int e = 0; e < DH; e++) acc[e] = fmaf(w, lv[e], acc[e]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&lv_free[g]);
            }
            if (!ok) break;
            {
                // rows 4 g + i of the lane group, chunk c = lane & 3 each (whole 64-byte runs);
                // rows past a packed sequence's end are not stored
                uint4 x[4];
#pragma unroll
                for (int c8 = 0; c8 < 4; c8++)
                    x[c8] = make_uint4(pack_bf16(acc[8 * c8], acc[8 * c8 + 1]), pack_bf16(acc[8 * c8 + 2], acc[8 * c8 + 3]),
                                       pack_bf16(acc[8 * c8 + 4], acc[8 * c8 + 5]), pack_bf16(acc[8 * c8 + 6], acc[8 * c8 + 7]));
                lane_group_transpose(x, lane);
                const int tg = q32 + (lane & ~3);
#pragma unroll
                for (int i = 0; i < 4; i++)
                    if (tg + i < live)
                        *reinterpret_cast<uint4*>(out + static_cast<size_t>(row0 + tg + i) * DV + half * DH + 8 * (lane & 3)) = x[i];
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------ host side

// Segment size 2^q: the node kernel keeps q level accumulators of dv/2 floats per
// thread in registers, within the 128 registers that let two CTAs share an SM
// (q <= 2 for dv = 64, q <= 1 for dv = 128); prefer at least two CTAs per SM worth
// of segments.
int choose_q(int BH, int NT, int dv) {
    const int qmax = dv == 64 ? 2 : 1;
    int q = 0;
    while (q < qmax && static_cast<int64_t>(BH) * ((NT + (2 << q) - 1) / (2 << q)) >= 2 * 152) q++;
    return q;
}


// tc_nodes + tc_merge: tile decays, the Fenwick nodes that are read (bf16), the per-token
// decay tables and the per-tile level decay table.
template <int DV>
cudaError_t tc_node_stage(const TcPlan& pl, const CUtensorMap& tk, const CUtensorMap& tv, const float* log_a,
                          void* workspace, int* err, cudaStream_t stream, const SeqMap& sm) {
    const int BH = pl.B * pl.H;
    const int qlog = pl.q;
    const int seg_tiles = 1 << qlog;
    const int nseg = (pl.NT + seg_tiles - 1) / seg_tiles;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* g_tiles = reinterpret_cast<float*>(ws);
    __nv_bfloat16* nodes = reinterpret_cast<__nv_bfloat16*>(ws + pl.g_bytes);
    float* seg_tot = reinterpret_cast<float*>(ws + pl.g_bytes + pl.nodes_bytes);
    float* dtab = reinterpret_cast<float*>(ws + pl.g_bytes + pl.nodes_bytes + pl.seg_bytes);
    float* tok_cl2 = reinterpret_cast<float*>(ws + pl.g_bytes + pl.nodes_bytes + pl.seg_bytes + pl.dtab_bytes);
    float* tok_colw = tok_cl2 + static_cast<size_t>(BH) * pl.T;
    int* tile_counter = reinterpret_cast<int*>(ws + pl.total_bytes - pl.ctr_bytes);
    LevelOffsets lo;
    for (int p = 0; p < 32; p++) lo.off[p] = pl.level_off[p];
    {
        const int smem = NodesSmem<DV>::kBytes;
        auto launch = [&](auto kern) -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            kern<<<dim3(nseg, BH), 256, smem, stream>>>(tk, tv, log_a, g_tiles, nodes, seg_tot, tok_cl2, tok_colw, pl.T,
                                                        pl.NT, pl.node_count, lo, sm, tile_counter, err);
            return cudaSuccess;
        };
        cudaError_t e;
        switch (qlog) {
            case 0: e = launch(tc_nodes_kernel<DV, 0>); break;
            case 1: e = launch(tc_nodes_kernel<DV, 1>); break;
            default: e = launch(tc_nodes_kernel<DV, DV == 64 ? 2 : 1>); break;
        }
        if (e != cudaSuccess) return e;
        note_launch(stream, "tc_nodes");
    }
    {
        const int msz = kDk * DV;
        int n_above = 0;
        for (int p = qlog + 1; p < pl.P; p++) n_above += (((pl.NT - 1) >> p) + 1) / 2;
        const cudaError_t e = launch_pdl(tc_merge_kernel, dim3(msz / 1024 + 1, n_above > 0 ? n_above : 1, BH), dim3(256),
                                         pl.NT * sizeof(float), stream, seg_tot, g_tiles, nodes, dtab, tile_counter,
                                         pl.NT, qlog, pl.P, nseg, pl.node_count, msz, lo, pl.T, sm);
        if (e != cudaSuccess) return e;
        note_launch(stream, "tc_merge");
    }
    return cudaGetLastError();
}

template <int DV>
cudaError_t tc_forward_dv(const TcPlan& pl, const void* q, const void* k, const void* v, const float* log_a,
                          const float* lambda, void* out, void* workspace, int* err, cudaStream_t stream,
                          bool nodes_only = false, SeqMap sm = SeqMap{nullptr, nullptr, 1, 0, 0}, int lam_levels = 0) {
    const int BH = pl.B * pl.H;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    __nv_bfloat16* nodes = reinterpret_cast<__nv_bfloat16*>(ws + pl.g_bytes);
    float* dtab = reinterpret_cast<float*>(ws + pl.g_bytes + pl.nodes_bytes + pl.seg_bytes);
    float* tok_cl2 = reinterpret_cast<float*>(ws + pl.g_bytes + pl.nodes_bytes + pl.seg_bytes + pl.dtab_bytes);
    float* tok_colw = tok_cl2 + static_cast<size_t>(BH) * pl.T;
    int* tile_counter = reinterpret_cast<int*>(ws + pl.total_bytes - pl.ctr_bytes);
    LevelOffsets lo;
    for (int p = 0; p < 32; p++) lo.off[p] = pl.level_off[p];
    if (!sm.seq) sm = SeqMap{nullptr, nullptr, pl.H, pl.B, 0};
    // input rows: [B*H*T] dense, [H * total_T] packed
    const uint64_t rows = sm.seq ? static_cast<uint64_t>(pl.H) * sm.total_T : static_cast<uint64_t>(BH) * pl.T;

    CUtensorMap tq, tk, tv, tn;
    if (!make_map(&tq, q, rows, pl.dk) || !make_map(&tk, k, rows, pl.dk) || !make_map(&tv, v, rows, DV))
        return cudaErrorInvalidValue;
    const bool have_nodes = pl.node_count > 0;
    if (have_nodes && !make_map(&tn, nodes, static_cast<uint64_t>(BH) * pl.node_count * kDk, DV))
        return cudaErrorInvalidValue;
    if (!have_nodes) tn = tv;  // never read when no tile has an earlier tile

    {
        cudaError_t e = tc_node_stage<DV>(pl, tk, tv, log_a, workspace, err, stream, sm);
        if (e != cudaSuccess || nodes_only) return e;
    }
    {
        // lambda row length: num_levels(T) dense; packed, that of the longest sequence (given)
        const int L = lam_levels > 0 ? lam_levels : bitlength(static_cast<int64_t>(pl.T) - 1) + 1;
        const int total = BH * pl.NT;
        const int grid = total < pl.num_sms ? total : pl.num_sms;
        if constexpr (DV == 64) {
            const int smem = PpCfg::kBytes;
            cudaError_t e =
                cudaFuncSetAttribute(tc_output_pp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            e = launch_pdl(tc_output_pp_kernel, dim3(grid), dim3(PpCfg::kThreads), smem, stream, tq, tk, tv, tn,
                           tok_cl2, tok_colw, lambda, dtab, static_cast<__nv_bfloat16*>(out), pl.T, pl.NT, L, pl.P,
                           pl.node_count, lo, total, tile_counter, sm, static_cast<int>(rows), err);
            if (e != cudaSuccess) return e;
        } else {
            const int smem = OutCfg<DV>::kBytes;
            cudaError_t e =
                cudaFuncSetAttribute(tc_output_kernel<DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            e = launch_pdl(tc_output_kernel<DV>, dim3(grid), dim3(OutCfg<DV>::kThreads), smem, stream, tq, tk, tv,
                           tn, tok_cl2, tok_colw, lambda, dtab, static_cast<__nv_bfloat16*>(out), pl.T, pl.NT, L,
                           pl.P, pl.node_count, lo, total, tile_counter, err);
            if (e != cudaSuccess) return e;
        }
        note_launch(stream, "tc_output");
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t tc_set_debug_waits(long long limit_cycles, int hold) {
    const long long lim = limit_cycles > 0 ? limit_cycles : kWaitCycles;
    const int h = hold != 0;
    cudaError_t e = cudaMemcpyToSymbol(tc_pipe_wait_limit, &lim, sizeof(lim));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(tc_debug_hold, &h, sizeof(h));
    return e;
}

bool tc_supported(int dtype, int dk, int dv, int T) {
    return dtype == 0 && (dk == 64 || dk == kDk) && (dv == 64 || dv == 128) && T % kTile == 0;
}

bool make_tc_plan(int B, int H, int T, int dk, int dv, TcPlan* pl) {
    pl->B = B; pl->H = H; pl->T = T; pl->dk = dk; pl->dv = dv;
    pl->NT = T / kTile;
    {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
            cudaGetLastError();
            sms = 152;
        }
        pl->num_sms = sms;
    }
    pl->P = bitlength(static_cast<int64_t>(pl->NT) - 1);
    const int BH = B * H;
    pl->q = choose_q(BH, pl->NT, dv);
    int off = 0;
    for (int p = 0; p < 32; p++) {
        pl->level_off[p] = off;
        if (p < pl->P) off += (((pl->NT - 1) >> p) + 1) / 2;  // even m with (m + 1) 2^p < NT
    }
    pl->node_count = off;
    const int seg_tiles = 1 << pl->q;
    const int nseg = (pl->NT + seg_tiles - 1) / seg_tiles;
    // 32-bit TMA row coordinates, a 16-entry level list per tile, merge totals in shared memory
    if (static_cast<int64_t>(BH) * T >= (int64_t(1) << 31) || pl->P > 16 || nseg > 12288) return false;
    if (pl->P - 1 - pl->q > 10) return false;  // the merge kernel weighs at most 1024 segments per node
    if (pl->NT > 8192) return false;            // and holds a head's tile totals in shared memory
    if (static_cast<int64_t>(BH) * pl->node_count * kDk >= (int64_t(1) << 31)) return false;
    const size_t msz = static_cast<size_t>(kDk) * dv;  // nodes are 128 x dv (dk = 64 pads rows 64..127)
    pl->g_bytes = (static_cast<size_t>(BH) * pl->NT * sizeof(float) + 1023) / 1024 * 1024;
    pl->nodes_bytes = (static_cast<size_t>(BH) * pl->node_count * msz * 2 + 1023) / 1024 * 1024;
    pl->seg_bytes = (static_cast<size_t>(BH) * nseg * msz * sizeof(float) + 1023) / 1024 * 1024;
    pl->dtab_bytes = static_cast<size_t>(BH) * pl->NT * 16 * sizeof(float);
    pl->tok_bytes = (2 * static_cast<size_t>(BH) * T * sizeof(float) + 255) / 256 * 256;
    pl->ctr_bytes = 256;
    pl->total_bytes = pl->g_bytes + pl->nodes_bytes + pl->seg_bytes + pl->dtab_bytes + pl->tok_bytes + pl->ctr_bytes;
    return true;
}

cudaError_t tc_forward(const TcPlan& pl, const void* q, const void* k, const void* v, const float* log_a,
                       const float* lambda, void* out, void* workspace, int* err, cudaStream_t stream) {
    if (pl.dv == 64) return tc_forward_dv<64>(pl, q, k, v, log_a, lambda, out, workspace, err, stream);
    return tc_forward_dv<128>(pl, q, k, v, log_a, lambda, out, workspace, err, stream);
}

bool tc_varlen_supported(int dtype, int dk, int dv) { return dtype == 0 && (dk == 64 || dk == kDk) && dv == 64; }

size_t tc_varlen_table_bytes(int n_seq) {
    return (static_cast<size_t>(n_seq) * sizeof(int2) + (n_seq + 1) * sizeof(int) + 255) / 256 * 256;
}

cudaError_t tc_forward_varlen(const TcPlan& pl, const void* q, const void* k, const void* v, const float* log_a,
                              const float* lambda, void* out, const int32_t* cu_seqlens, int total_T, int max_T,
                              int lam_levels, void* workspace, void* table, int* err, cudaStream_t stream) {
    if (pl.dv != 64) return cudaErrorInvalidValue;
    int2* seq = static_cast<int2*>(table);
    int* prefix = reinterpret_cast<int*>(seq + pl.B);
    seq_table_kernel<<<1, 1024, 0, stream>>>(cu_seqlens, seq, prefix, pl.B, pl.H, total_T, max_T, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    note_launch(stream, "seq_table");
    return tc_forward_dv<64>(pl, q, k, v, log_a, lambda, out, workspace, err, stream, false,
                             SeqMap{seq, prefix, pl.H, pl.B, total_T}, lam_levels);
}

cudaError_t tc_nodes_only(const TcPlan& pl, const void* k, const void* v, const float* log_a, void* workspace,
                          int* err, cudaStream_t stream) {
    if (pl.dv == 64) return tc_forward_dv<64>(pl, k, k, v, log_a, nullptr, nullptr, workspace, err, stream, true);
    return tc_forward_dv<128>(pl, k, k, v, log_a, nullptr, nullptr, workspace, err, stream, true);
}

}  // namespace lla
