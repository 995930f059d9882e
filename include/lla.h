/*
 * lla.h — C ABI of liblla.so: causal log-linear Mamba-2 attention on GB300 (sm_103a).
 *
 * The operator ("Log-Linear Attention", arXiv 2506.04761; gist.science pages in
 * Portuguese and French, §2 "Particionamento Hierarquico / Mascara Hierarquica"
 * and "Partitionnement par Arbre de Fenwick / Matrice de Masque Hierarchique"):
 *
 *     O = (Q K^T (.) M^S (.) M^H) V
 *     o_t = sum_{s<=t} lambda_t^(l(t,s)) * prod_{r=s+1..t} a_r * (q_t . k_s) * v_s
 *
 * M^S is the Mamba-2 semiseparable scalar-decay mask (a_r = exp(log_a_r) in
 * (0,1], exclusive of s so the diagonal is 1). M^H weights key s for query t
 * by lambda_t at the Fenwick level l(t,s) of s in t's prefix: l = 0 for s = t,
 * otherwise the bucket of size 2^(l-1) in the Fenwick decomposition of [0,t),
 * which equals 1 + floor(log2(t xor s)) with 0-indexed positions. A length-T
 * sequence uses L = bitlength(T-1) + 1 levels (7, 12, 14, 17 for T = 64, 2048,
 * 8192, 65536). There is no 1/sqrt(d) scale and no normalisation.
 *
 * Conventions for every entry point:
 *  - Tensors are dense, row-major (C-contiguous), batch-major: [B, H, ...].
 *  - q/k/v/out are bf16 (LLA_BF16) or fp32 (LLA_F32); log_a, lambda and decode
 *    states are always fp32; decode positions are int64.
 *  - Device pointers are caller-owned CUDA device memory on the current device.
 *    The library keeps no pointer after the call returns. Every pointer must be
 *    16-byte aligned.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). All work is
 *    enqueued asynchronously on it; outputs are valid once the stream reaches
 *    that point.
 *  - Return value: LLA_OK, or a negative lla_status. Argument errors are found
 *    on the host before anything is enqueued and leave all buffers untouched.
 *    Faults found by a kernel (an out-of-range decode position, a bounded wait
 *    that ran out) are recorded in a per-device error word and reported by
 *    lla_device_error(). No kernel traps and the library never exits.
 *  - The library keeps per-device state for the life of the process: the device
 *    address of its error word and of the lla_forward_noalloc scratch, looked up
 *    once, and a memory pool. Do not call it on a device after cudaDeviceReset()
 *    (or any teardown of that device's primary context) in the same process: the
 *    cached addresses would no longer be valid.
 */
#ifndef LLA_H
#define LLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LLA_OK = 0,
    LLA_ERR_INVALID_ARG = -1, /* null pointer, bad size, misaligned pointer */
    LLA_ERR_UNSUPPORTED = -2, /* valid operator, but a shape this build has no kernel for */
    LLA_ERR_CUDA = -3,        /* a CUDA runtime call or launch failed */
    LLA_ERR_TIMEOUT = -4,     /* a kernel's bounded wait ran out (device error word) */
    LLA_ERR_NOMEM = -5,       /* workspace allocation failed, or workspace too small */
    LLA_ERR_DEVICE = -6       /* a kernel rejected its device-side input (device error word) */
} lla_status;

typedef enum { LLA_BF16 = 0, LLA_F32 = 1 } lla_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char* lla_status_string(int status);

/* Number of Fenwick levels used by a length-T sequence: bitlength(T-1) + 1
 * (1 for T = 1, 0 for T <= 0). lambda's last dimension must equal this. */
int lla_num_levels(int64_t T);

/*
 * Chunk-parallel prefill (pages' "Chunk-scan" / "balayage par blocs": dense
 * intra-chunk work, hierarchical inter-chunk state passing, O(T log T)).
 *
 *   q      [B,H,T,dk]  dtype        queries
 *   k      [B,H,T,dk]  dtype        keys
 *   v      [B,H,T,dv]  dtype        values
 *   log_a  [B,H,T]     fp32         log of the Mamba-2 decay a_t (<= 0 expected;
 *                                   positive values are computed as given)
 *   lambda [B,H,T,L]   fp32         per-query, per-level weights, L = lla_num_levels(T)
 *   out    [B,H,T,dv]  dtype        written; must not overlap any input
 *   chunk  chunk length of the scan: 16, 32, 64 or 128, with T % chunk == 0.
 *          It sets how keys are grouped into inter-chunk states; the result is
 *          the same operator for every valid chunk (up to rounding order).
 *   dk, dv 1..128; the bf16 tensor-core path runs for dk in {64,128}, dv in {64,128},
 *          T % 128 == 0; other shapes run the fp32 SIMT path.
 *
 * Scratch: the call takes its workspace (inter-chunk states) from a
 * library-owned, stream-ordered memory pool on `stream` and returns it there.
 * Use lla_forward_ws to pass caller-owned workspace instead.
 */
int lla_forward(const void* q, const void* k, const void* v, const float* log_a, const float* lambda,
                void* out, int B, int H, int T, int dk, int dv, int chunk, void* stream, int dtype);

/*
 * lla_forward with HOST buffers (pinned for full copy bandwidth; pageable works,
 * slower): same arguments and layouts as lla_forward, but q, k, v, log_a, lambda
 * and out live in host memory (device or managed pointers: LLA_ERR_INVALID_ARG).
 * The B*H heads are split into up to eight groups; each group's inputs are copied
 * to the device on a library copy stream, its prefill runs on `stream`, and its
 * output is copied back on a second library stream, so copies of one group
 * overlap the kernels of the next. Device buffers come from the library pool.
 * The call returns after `out` is written (it synchronizes `stream`). Calls on
 * one device are serialized.
 */
int lla_forward_host(const void* q, const void* k, const void* v, const float* log_a, const float* lambda,
                     void* out, int B, int H, int T, int dk, int dv, int chunk, void* stream, int dtype);

/* Workspace bytes lla_forward_ws needs for these sizes (0 on invalid sizes). */
size_t lla_forward_workspace_size(int B, int H, int T, int dk, int dv, int chunk, int dtype);

/* lla_forward with caller-owned device workspace of at least
 * lla_forward_workspace_size(...) bytes, 256-byte aligned. The workspace holds
 * no state between calls; calls that share it must not overlap on the GPU.
 * Returns LLA_ERR_NOMEM if workspace_bytes is too small. */
int lla_forward_ws(const void* q, const void* k, const void* v, const float* log_a, const float* lambda,
                   void* out, int B, int H, int T, int dk, int dv, int chunk, void* stream, int dtype,
                   void* workspace, size_t workspace_bytes);

/*
 * lla_forward without any allocation, for callers that cannot call cudaMalloc
 * (a host that pre-sizes and owns every device allocation, or code that must
 * not grow the process's GPU footprint after start-up). "Log-Linear Attention"
 * describes no counterpart: this is a deployment variant of lla_forward with
 * identical arguments, results and kernels.
 *
 * Its scratch is a fixed, file-scope device array of LLA_NOALLOC_SCRATCH_BYTES
 * (32 MiB) that every GPU loading this library holds until the process exits.
 * Sizes whose workspace (lla_forward_workspace_size) exceeds it are rejected
 * with LLA_ERR_NOMEM before anything is enqueued. No cudaMalloc, cudaFree or
 * allocating library routine is called.
 *  - The first call on a device looks up that device's copy of the array; make
 *    that first call before capturing a stream into a CUDA graph. The address is
 *    kept for the life of the process (see the cudaDeviceReset note above).
 *  - Every call on a device shares the one array and leaves its contents
 *    behind; no part of it needs to start at zero (each call writes every
 *    scratch value before reading it). Calls whose work overlaps on the GPU
 *    (different streams, or graphs replayed concurrently) race on the array:
 *    serialise them.
 */
#define LLA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int lla_forward_noalloc(const void* q, const void* k, const void* v, const float* log_a, const float* lambda,
                        void* out, int B, int H, int T, int dk, int dv, int chunk, void* stream, int dtype);

/*
 * Measurement aid: runs lla_forward once with a CUDA event recorded on `stream`
 * before the first kernel and after each kernel launch, waits for the last
 * event, and writes, in launch order, each kernel's elapsed device time in
 * milliseconds to kernel_ms[i] and its static name to kernel_names[i], for
 * i < cap. Returns the number of kernels the call launched (which may exceed
 * cap), or a negative lla_status. Synchronous; not meant for hot loops.
 */
int lla_forward_profile(const void* q, const void* k, const void* v, const float* log_a, const float* lambda,
                        void* out, int B, int H, int T, int dk, int dv, int chunk, void* stream, int dtype,
                        float* kernel_ms, const char** kernel_names, int cap);

/*
 * One recurrent decode step (pages' "Decodificacao" / "Inference": O(log T)
 * states S_t^(l), the new token updates the finest level and levels merge
 * along the Fenwick tree; O(log T) time and memory per step).
 *
 *   q, k   [B,H,dk]          dtype   the new token's query and key
 *   v      [B,H,dv]          dtype   its value
 *   log_a  [B,H]             fp32    log a_t of the new token
 *   lambda [B,H,Lmax]        fp32    lambda_t^(l) of the new token, l < Lmax
 *   fenwick_states [B,H,Lmax,dk,dv] fp32, read and written in place.
 *          Slot l holds bucket l of the Fenwick partition as
 *          sum_s prod_{r=s+1..pos} a_r k_s v_s^T, decayed to the last token
 *          `pos` already absorbed. On entry pos = t[b]-1 (nothing for t[b] = 0);
 *          on return pos = t[b]. Slots empty at `pos` (level l >= 1 with bit
 *          l-1 of pos clear) are never read and may hold anything.
 *   t      [B]               int64   device array: position of the new token per
 *          sequence (tokens 0..t-1 are in the states). Not modified: the caller
 *          advances it. Needs 0 <= t < 2^(Lmax-1); a sequence outside that range
 *          is skipped (its state and output untouched) and LLA_ERR_DEVICE is
 *          recorded in the device error word.
 *   out    [B,H,dv]          dtype   o_t = sum_l lambda_t^(l) S^(l)^T q_t (after the update)
 *   dk     1..256; dv in {16, 32, 64, 128}; Lmax in 1..40.
 */
int lla_decode_step(const void* q, const void* k, const void* v, const float* log_a, const float* lambda,
                    float* fenwick_states, const int64_t* t, void* out, void* stream,
                    int B, int H, int dk, int dv, int Lmax, int dtype);

/*
 * Prefill -> decode hand-off: the Fenwick state set after a prompt of T tokens,
 * i.e. what lla_decode_step expects on entry for the next position t = T.
 *
 *   k      [B,H,T,dk]  dtype   keys of the prompt
 *   v      [B,H,T,dv]  dtype   values
 *   log_a  [B,H,T]     fp32    log decays
 *   fenwick_states [B,H,Lmax,dk,dv] fp32, written for every sequence: slot 0 =
 *          k_{T-1} v_{T-1}^T, and each slot l >= 1 with bit l-1 of T-1 set = its
 *          Fenwick bucket of T-1's prefix, sum_s prod_{r=s+1..T-1} a_r k_s v_s^T.
 *          Slots empty at T-1 are left untouched. Needs Lmax >= bitlength(T-1) + 1.
 *   dk, dv 1..128.
 * Takes T fp32 values per (b, h) of scratch from the library's stream-ordered pool.
 * Tensor-core path (bf16, dk = 128): every held slot is written exactly once, its
 * pieces summed in a fixed order, so repeated calls give identical bits. The
 * CUDA-core path adds bucket pieces of at most 512 keys with fp32 atomics, so for
 * buckets of more than 1024 keys the last bits may vary between runs.
 */
int lla_prefill_state(const void* k, const void* v, const float* log_a, float* fenwick_states, int B, int H, int T,
                      int dk, int dv, int Lmax, void* stream, int dtype);

/*
 * Backward of lla_forward: gradients of L = sum over all elements of dout * out.
 * ("Log-Linear Attention", pt §2 "Mascara Hierarquica" / fr §2 "Matrice de
 * Masque Hierarchique" define the operator differentiated here; the pages name
 * the backward through lambda as needing its own kernels.)
 *
 *   q, k, v, log_a, lambda   the forward's inputs (same shapes, dtype, chunk rules)
 *   dout     [B,H,T,dv]  dtype   upstream gradient dL/dout
 *   dq, dk   [B,H,T,dk]  dtype   written
 *   dv       [B,H,T,dv]  dtype   written
 *   dlog_a   [B,H,T]     fp32    written
 *   dlambda  [B,H,T,L]   fp32    written (0 for levels with no key at that query)
 * The outputs must not overlap any input or each other. The forward's
 * intermediate states are recomputed, so no forward workspace is kept between
 * the calls. The chunk argument follows lla_forward. bf16 inputs with dk = 128,
 * dv = 64 and T % 128 == 0 run on tensor cores (128-token tiles, fp32
 * accumulation, bf16 operands); every other shape runs fp32 arithmetic on CUDA
 * cores with chunks of at most 64 (chunk 128 runs as 64: same operator,
 * different rounding order). Workspace comes from the same library-owned
 * stream-ordered pool as lla_forward. A kernel's bounded wait that runs out is
 * reported by lla_device_error as LLA_ERR_TIMEOUT. Errors: LLA_ERR_INVALID_ARG / LLA_ERR_UNSUPPORTED before any
 * launch, LLA_ERR_NOMEM if the pool cannot grow, LLA_ERR_CUDA on launch
 * failure.
 */
int lla_backward(const void* q, const void* k, const void* v, const float* log_a, const float* lambda,
                 const void* dout, void* dq, void* dk, void* dv, float* dlog_a, float* dlambda, int B, int H,
                 int T, int dk_, int dv_, int chunk, void* stream, int dtype);

/*
 * Packed variable-length sequences (no counterpart on the pages: a serving
 * layout for many prompts of different lengths in one call).
 *
 * Layout: every tensor is packed per head, [H, total_T, W] row-major; sequence
 * b owns rows cu_seqlens[b] .. cu_seqlens[b+1]-1 of every head, and its token
 * positions (hence its Fenwick levels) start at 0. cu_seqlens is DEVICE int32
 * [n_seq + 1], non-decreasing, cu_seqlens[0] >= 0, cu_seqlens[n_seq] <= total_T,
 * every length <= max_T. Lengths that break these rules are caught on the
 * device: that sequence is skipped and lla_device_error reports LLA_ERR_DEVICE.
 *
 * lla_forward_varlen: the prefill of every sequence.
 *   q, k [H,total_T,dk], v [H,total_T,dv] (dtype); log_a [H,total_T] fp32;
 *   lambda [H,total_T,L] fp32 with L = lla_num_levels(max_T); out [H,total_T,dv].
 *   bf16 with dv = 64 and dk in {64, 128}: the tensor-core prefill kernels walk
 *   every sequence's own 128-token tiles of the packed tensors (a sequence's
 *   last tile may end inside it; its rows past the end are neither read into
 *   the sequence's outputs nor written). Other shapes: the sequences are copied
 *   into a zero-padded [n_seq, H, Tpad] layout (Tpad = max_T rounded up to
 *   128) in pool workspace, run through the dense prefill kernels and copied
 *   back. Requires H * total_T < 2^31 for the tensor-core walk. chunk as in
 *   lla_forward.
 *
 * lla_prefill_state_varlen: the decode state set after every sequence, as
 * lla_prefill_state: fenwick_states [n_seq, H, Lmax, dk, dv] fp32 with
 * Lmax >= lla_num_levels(max_T); slots empty at a sequence's last position are
 * left untouched (an empty sequence touches none). bf16 with dk = 128 and
 * dv in {64, 128} runs the tensor-core hand-off over every sequence's own tile
 * range; other shapes run CUDA-core kernels.
 */
int lla_forward_varlen(const void* q, const void* k, const void* v, const float* log_a, const float* lambda,
                       void* out, const int32_t* cu_seqlens, int n_seq, int H, int total_T, int max_T, int dk, int dv,
                       int chunk, void* stream, int dtype);
int lla_prefill_state_varlen(const void* k, const void* v, const float* log_a, const int32_t* cu_seqlens,
                             float* fenwick_states, int n_seq, int H, int total_T, int max_T, int dk, int dv, int Lmax,
                             void* stream, int dtype);

/*
 * Log-linear Gated DeltaNet ("Log-Linear Attention", pt §2 "Generalizacao" and
 * fr §3 "Etudes de Cas": the hierarchical mask applied to Gated DeltaNet; the
 * base model is Gated DeltaNet's published gated delta rule):
 *
 *     o_t = sum_{s<=t} lambda_t^(l(t,s)) A[t,s] v_s,
 *     A[t,s] = beta_s k_s^T A_{s+1} A_{s+2} ... A_t q_t,
 *     A_r = exp(log_a_r) (I - beta_r k_r k_r^T),
 *
 * i.e. Gated DeltaNet's own attention matrix under the Fenwick mask M^H. In
 * recurrent form every held Fenwick bucket state S (dk x dv) evolves as
 * S <- A_t S, buckets merge on the lowbit carry as in lla_decode_step, and the
 * new token writes beta_t k_t v_t^T at level 0. Keys are expected L2-normalised
 * and beta in [0, 1] (the transition is then a contraction); other values are
 * computed as given.
 *
 * lla_gdn_forward: chunkwise prefill. Arguments as lla_forward, plus
 *   beta   [B,H,T]  fp32   delta-rule strength of every token.
 *   chunk  16, 32, 64 or 128 (128 runs as 64: same operator, different rounding
 *          order), T % chunk == 0; dk 1..128; dv a multiple of 16 up to 128.
 * All arithmetic is fp32 on CUDA cores. Workspace comes from the library's
 * stream-ordered pool: per head about (2 dk T + 2 (T / C) dk dv + dv T) floats.
 *
 * lla_gdn_decode_step: one recurrent step; arguments as lla_decode_step, plus
 *   beta   [B,H]    fp32   the new token's delta-rule strength.
 *   fenwick_states holds each bucket's state under the transitions above (the
 *   layout, emptiness and position rules of lla_decode_step apply unchanged).
 *   dk and dv in {16, 32, 64, 128}.
 */
int lla_gdn_forward(const void* q, const void* k, const void* v, const float* log_a, const float* beta,
                    const float* lambda, void* out, int B, int H, int T, int dk, int dv, int chunk, void* stream,
                    int dtype);
int lla_gdn_decode_step(const void* q, const void* k, const void* v, const float* log_a, const float* beta,
                        const float* lambda, float* fenwick_states, const int64_t* t, void* out, void* stream, int B,
                        int H, int dk, int dv, int Lmax, int dtype);
/* Measurement aid for lla_gdn_forward, as lla_forward_profile is for lla_forward. */
int lla_gdn_forward_profile(const void* q, const void* k, const void* v, const float* log_a, const float* beta,
                            const float* lambda, void* out, int B, int H, int T, int dk, int dv, int chunk,
                            void* stream, int dtype, float* kernel_ms, const char** kernel_names, int cap);

/*
 * Test hook for the failure path of the bounded waits (no counterpart on the
 * pages; not for production use). On the current device, for the tensor-core
 * prefill output kernel of dv = 64: limit_cycles > 0 bounds each of its pipeline
 * waits to that many SM cycles (<= 0 restores the default, about 2 s at the
 * maximum clock); hold != 0 makes its epilogue first wait on a barrier that
 * nothing arrives at, so that wait runs out. The kernel then records
 * LLA_ERR_TIMEOUT in the device error word, lets its own in-flight copies and
 * MMAs land (those drain waits keep the full bound), frees its tensor memory and
 * returns; the call's output is then undefined. Synchronous with the host; takes
 * effect for kernels launched afterwards. Returns LLA_OK or LLA_ERR_CUDA.
 */
int lla_debug_set_waits(int64_t limit_cycles, int hold);

/*
 * Reads and clears the device error word of the current device after
 * synchronising `stream`: LLA_OK if no kernel recorded a fault since the last
 * read, LLA_ERR_DEVICE for rejected device-side input, LLA_ERR_TIMEOUT for a
 * bounded wait that ran out, LLA_ERR_CUDA if the synchronisation itself failed.
 */
int lla_device_error(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LLA_H */
