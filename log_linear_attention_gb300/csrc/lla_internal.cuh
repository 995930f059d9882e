// Internal declarations shared by the host API (lla_api.cu) and the kernel
// translation units. Not part of the public ABI (see include/lla.h).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

namespace lla {

// Device error word values (a kernel writes the first fault it sees with atomicCAS).
enum DeviceError : int { kDevOk = 0, kDevBadInput = 1, kDevTimeout = 2 };

__device__ __forceinline__ void record_error(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ float load_f(const float* p) { return *p; }
__device__ __forceinline__ float load_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void store_f(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_f(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// Fenwick level of key s for query t (s <= t), 0-indexed positions:
// 0 for s == t, else 1 + floor(log2(t xor s)). Valid for positions < 2^31.
__device__ __forceinline__ int fenwick_level(int t, int s) { return 32 - __clz(t ^ s); }

// Optional per-launch event log for lla_forward_profile: when a log is active on
// this host thread, every launcher calls note_launch() right after enqueueing a
// kernel, which records a CUDA event on the launch stream.
struct LaunchLog {
    static constexpr int kMax = 32;
    cudaEvent_t events[kMax];
    const char* names[kMax];
    int count;
};
LaunchLog*& active_launch_log();
inline void note_launch(cudaStream_t stream, const char* name) {
    LaunchLog* log = active_launch_log();
    if (!log) return;
    if (log->count < LaunchLog::kMax) {
        log->names[log->count] = name;
        cudaEventRecord(log->events[log->count], stream);
    }
    log->count++;
}

inline int bitlength(int64_t x) {
    int n = 0;
    while (x > 0) { n++; x >>= 1; }
    return n;
}

// Layout of the SIMT path's workspace for one lla_forward call.
//   g      fp32 [BH][N]                        per-chunk total log-decay
//   nodes  fp32 [BH][node_count][dk][dv]      Fenwick pyramid: level p holds
//          N >> p nodes; node (p, m) is the decayed state sum of chunks
//          [m 2^p, (m+1) 2^p), decayed to the last token of the block.
struct SimtPlan {
    int B, H, T, dk, dv, chunk, c;  // c = log2(chunk)
    int N;                          // chunks per sequence
    int P;                          // pyramid levels read: bitlength(N - 1)
    int node_count;                 // sum_{p<P} N >> p
    int level_off[32];              // first node of level p
    size_t g_bytes, nodes_bytes, total_bytes;
};

bool make_simt_plan(int B, int H, int T, int dk, int dv, int chunk, SimtPlan* plan);

// Tensor-core (tcgen05) path for bf16, dk = 128. Plan and launcher live in lla_tc.cu.
struct TcPlan {
    int B, H, T, dk, dv;
    int NT;                  // 128-token tiles per sequence
    int P;                   // node levels read: bitlength(NT - 1)
    int q;                   // log2 of the tiles per segment of the node kernel
    int num_sms;             // persistent grid size of the output kernel
    int node_count;          // even-indexed nodes actually read, all levels
    int level_off[32];       // node index of (p, m = 0); node (p, m even) at level_off[p] + m / 2
    size_t g_bytes, nodes_bytes, seg_bytes, dtab_bytes, tok_bytes, ctr_bytes, total_bytes;
};

bool tc_supported(int dtype, int dk, int dv, int T);
bool make_tc_plan(int B, int H, int T, int dk, int dv, TcPlan* plan);
cudaError_t tc_forward(const TcPlan& plan, const void* q, const void* k, const void* v, const float* log_a,
                       const float* lambda, void* out, void* workspace, int* err, cudaStream_t stream);
// Packed variable-length sequences (bf16, dv = 64, dk in {64, 128}) on the tensor-core kernels:
// plan = make_tc_plan(n_seq, H, Tpad = max_T rounded up to 128, dk, dv); tensors [H, total_T, .];
// `table` holds tc_varlen_table_bytes(n_seq) of device scratch (the validated sequence table).
bool tc_varlen_supported(int dtype, int dk, int dv);
size_t tc_varlen_table_bytes(int n_seq);
cudaError_t tc_forward_varlen(const TcPlan& plan, const void* q, const void* k, const void* v, const float* log_a,
                              const float* lambda, void* out, const int32_t* cu_seqlens, int total_T, int max_T,
                              int lam_levels, void* workspace, void* table, int* err, cudaStream_t stream);
// Failure-path test hooks of the dv = 64 output kernel on the current device: the bound
// on its pipeline waits (limit_cycles <= 0: the default of about 2 s) and a wait that
// nothing completes (hold != 0).
cudaError_t tc_set_debug_waits(long long limit_cycles, int hold);
// The node stage of tc_forward only (tc_nodes + tc_merge), for the backward.
cudaError_t tc_nodes_only(const TcPlan& plan, const void* k, const void* v, const float* log_a, void* workspace,
                          int* err, cudaStream_t stream);

// Tensor-core state set after a prefill (lla_tc_state.cu): bf16, dk = 128, dv in {64, 128}.
// Dense: B sequences of T rows. Packed (cu non-null, device int32 [B+1]): sequence b of head h
// has cu[b+1] - cu[b] <= T rows starting at row h * total + cu[b].
bool tc_state_supported(int dtype, int dk, int dv, int B, int H, int T);
bool tc_state_supported_packed(int dtype, int dk, int dv, int n_seq, int H, int total, int max_T);
size_t tc_state_workspace_bytes(int B, int H, int T, int dv);
cudaError_t tc_prefill_state(const void* k, const void* v, const float* log_a, float* states, int B, int H, int T,
                             int dv, int Lmax, void* workspace, int* err, cudaStream_t stream,
                             const int32_t* cu = nullptr, int total = 0);

// SIMT launchers (lla_simt.cu).
cudaError_t simt_forward(const SimtPlan& plan, int dtype, const void* q, const void* k, const void* v,
                         const float* log_a, const float* lambda, void* out, void* workspace, int* err,
                         cudaStream_t stream);
// CUDA-core state set after a prefill. Dense: B sequences of T rows each. Packed (cu_seqlens
// non-null, device int32 [B+1]): sequence b of head h has cu[b+1] - cu[b] <= T rows starting
// at row h * total + cu[b]. Workspace: one float per row.
cudaError_t prefill_state(int dtype, const void* k, const void* v, const float* log_a, float* states, int B, int H,
                          int T, int dk, int dv, int Lmax, void* workspace, int* err, cudaStream_t stream,
                          const int32_t* cu_seqlens = nullptr, int total = 0);
// The first half of the SIMT forward: chunk totals g and every fp32 pyramid node, laid out as
// SimtPlan describes at the start of `workspace`.
cudaError_t simt_nodes(const SimtPlan& plan, int dtype, const void* k, const void* v, const float* log_a,
                       void* workspace, cudaStream_t stream);

// Backward (lla_bwd.cu): plan and launcher.
struct BwdPlan {
    SimtPlan fw;             // forward nodes recomputed with the backward's chunk
    int n_read;              // read nodes (p, m even, (m + 1) 2^p < N), all levels
    int read_off[32];        // first read node of level p
    int max_pieces;          // token pieces of the largest query block
    size_t dnodes_bytes, dcum_bytes, total_bytes;
};
bool make_bwd_plan(int B, int H, int T, int dk, int dv, int chunk, BwdPlan* plan);
cudaError_t simt_backward(const BwdPlan& plan, int dtype, const void* q, const void* k, const void* v,
                          const float* log_a, const float* lambda, const void* dout, void* dq, void* dk, void* dv,
                          float* dlog_a, float* dlambda, void* workspace, cudaStream_t stream);
// Packed <-> padded copies for variable-length sequences (lla_varlen.cu); elem_bytes 2 = bf16, 4 = fp32.
cudaError_t varlen_pack(int elem_bytes, const void* src, void* dst, const int32_t* cu, int n_seq, int H, int total,
                        int Tpad, int W, int Wp, int max_len, int* err, cudaStream_t stream);
cudaError_t varlen_unpack(int elem_bytes, const void* src, void* dst, const int32_t* cu, int n_seq, int H, int total,
                          int Tpad, int W, int max_len, int* err, cudaStream_t stream);

// dlog_a_r = sum_{t >= r} dcum_t per head (lla_bwd.cu).
cudaError_t bwd_dloga(const float* dcum, float* dlog_a, int BH, int T, cudaStream_t stream);

// Tensor-core backward (lla_tc_bwd.cu): bf16, dk = 128, dv = 64, T % 128 == 0.
bool tc_bwd_supported(int dtype, int dk, int dv, int T);
size_t tc_bwd_workspace_bytes(const TcPlan& plan);
cudaError_t tc_backward(const TcPlan& plan, const void* q, const void* k, const void* v, const float* log_a,
                        const float* lambda, const void* dout, void* dq, void* dk, void* dv, float* dlog_a,
                        float* dlambda, void* workspace, int* err, cudaStream_t stream);
// Log-linear Gated DeltaNet (lla_gdn.cu): chunkwise prefill on CUDA cores and the decode step.
struct GdnPlan {
    int B, H, T, dk, dv;
    int C;                   // chunk of the scan (the API chunk, at most 64)
    int N;                   // chunks per sequence
    int P;                   // node levels read: bitlength(N - 1)
    int node_count;          // complete nodes per head, all levels <= P
    int level_off[32];       // first node of level p
    size_t w_off, qt_off, node_off, gam_off, oacc_off, total_bytes;
};
bool make_gdn_plan(int B, int H, int T, int dk, int dv, int chunk, GdnPlan* plan);
cudaError_t gdn_forward(const GdnPlan& plan, int dtype, const void* q, const void* k, const void* v,
                        const float* log_a, const float* beta, const float* lambda, void* out, void* workspace,
                        int* err, cudaStream_t stream);
// Tensor-core chunk and level passes (bf16, C = 64, dv = 64, dk in {64, 128}); csrc/lla_gdn_tc.cu.
bool gdn_chunk_tc_supported(const GdnPlan& plan, int dtype);
cudaError_t gdn_chunk_tc(const GdnPlan& plan, const void* q, const void* k, const void* v, const float* log_a,
                         const float* beta, const float* lambda, float* Wg, float* Qt, float* nodes, float* gam,
                         float* oacc, void* out, int L, int* err, cudaStream_t stream);
bool gdn_level_tc_supported(const GdnPlan& plan, int dtype);
cudaError_t gdn_levels_tc(const GdnPlan& plan, const void* k, const float* Wg, const float* Qt, float* nodes,
                          const float* gam, const float* lambda, float* oacc, int L, int c_log2, int* err,
                          cudaStream_t stream);
cudaError_t gdn_decode_step(int dtype, const void* q, const void* k, const void* v, const float* log_a,
                            const float* beta, const float* lambda, float* states, const int64_t* t, void* out, int B,
                            int H, int dk, int dv, int Lmax, int* err, cudaStream_t stream);

cudaError_t decode_step(int dtype, const void* q, const void* k, const void* v, const float* log_a,
                        const float* lambda, float* states, const int64_t* t, void* out, int B, int H,
                        int dk, int dv, int Lmax, int* err, cudaStream_t stream);

}  // namespace lla
