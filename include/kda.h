/*
 * kda.h -- C ABI of the Kimi Delta Attention (KDA) library for one GB300 (sm_103a).
 *
 * KDA is a gated delta rule with channel-wise decay.  Per (sequence, head) it
 * carries a key-by-value state S (dk x dv, fp32) and, for each token t,
 *
 *     S_t = (I - beta_t k_t k_t^T) . Diag(exp g_t) . S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t
 *
 * Sources (Kimi K3 report as summarised on the llm-atlas page "K3_RESEARCH.md"):
 * question ledger Q04 (fixed-shape recurrent state, channel-wise decay,
 * delta-rule write), Q05 (the write subtracts the state's prediction for the
 * current key), Q06 and Figure 3 (log-decay bounded below by g_min = -5 so the
 * diagonal tile can use BF16 tensor-core matmuls), Q07 (chunkwise-parallel
 * prefill with the state passed between chunks; O(1) state update for decode),
 * Q10 (attention output kept in FP32), and section 8's device layer ("fused
 * decode").  The agihunt digest page adds that FlashKDA cuts chunks further into
 * 16-token tiles for numerical stability.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are caller-owned DEVICE memory of the current CUDA
 *     device, contiguous, 16-byte aligned (beta and cu_seqlens: 4-byte
 *     aligned) -- except for kda_prefill_host and kda_prefill_host_static, whose
 *     tensors are HOST memory.  The library allocates no memory per call: the
 *     host-buffer path creates its streams and events once per device, and
 *     kda_prefill_host_static's scratch is a fixed array in the library's image.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Work is enqueued asynchronously on it; the call returns at once.
 *   - Argument errors are detected on the host and returned synchronously,
 *     before anything is enqueued.  A failed launch returns KDA_ERR_CUDA.
 *   - Errors found on the device (a bad cu_seqlens entry, a bounded wait that
 *     gave up) are recorded in a per-device status word; the affected work is
 *     skipped, nothing traps.  kda_last_device_status() reports and clears it.
 *   - q is not scaled (no 1/sqrt(dk)); callers pre-scale q if they want that.
 *   - Input prologue (the `prologue` word of kda_prefill_desc, kda_decode and
 *     kda_decode_multi; 0 = the inputs are used as given).  The workloads'
 *     input recipe -- q and k L2-normalised per (token, head), g = g_min *
 *     sigmoid(.), beta = sigmoid(.) -- can run inside the kernels' loads instead
 *     of as separate passes over HBM:
 *       KDA_PROLOGUE_QK_L2NORM   q and k are replaced by x / max(||x||_2, 1e-12)
 *                                over the dk channels of each (token, head),
 *                                computed in fp32 and rounded to qkv_dtype;
 *       KDA_PROLOGUE_G_LOGITS    g holds logits z; the decay used is -5 * sigmoid(z);
 *       KDA_PROLOGUE_BETA_LOGITS beta holds logits y; the write used is sigmoid(y).
 *   - Output gate (kda_prefill_gated, kda_decode_gated, kda_decode_multi_gated):
 *     the pages give KDA an input-dependent, full-rank gate over the read-out
 *     channels (llm-atlas Q08) but not its formula.  This library reads it as an
 *     elementwise sigmoid gate applied to the fp32 output, out = o * sigmoid(z),
 *     with the logits z [.., H, dv] fp32 computed by the caller (the projection
 *     that produces them is outside the attention kernel).  The gate changes only
 *     the written output, never the state.
 *   - Preconditions not checked on the host: g in [-5, 0] (the bounded
 *     log-decay; never clamped), beta in [0, 1].  Values outside these ranges
 *     are unsupported: they are computed, but without the accuracy bound.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_ABI_VERSION 3

#define KDA_PROLOGUE_QK_L2NORM 1
#define KDA_PROLOGUE_G_LOGITS 2
#define KDA_PROLOGUE_BETA_LOGITS 4
#define KDA_PROLOGUE_ALL 7

typedef enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = -1,   /* null/misaligned pointer, bad size, aliasing, bad cu_seqlens */
    KDA_ERR_UNSUPPORTED = -2,   /* head dims other than dk == dv in {64, 128}, unknown dtype */
    KDA_ERR_WORKSPACE = -3,     /* workspace smaller than kda_prefill_workspace_bytes() */
    KDA_ERR_CUDA = -4,          /* a CUDA runtime call or kernel launch failed */
    KDA_ERR_TIMEOUT = -5        /* a bounded on-device wait gave up (work skipped) */
} kda_status;

/* Storage type of q, k, v.  g, beta, states and outputs are always fp32. */
typedef enum kda_dtype {
    KDA_F32 = 0,
    KDA_BF16 = 1
} kda_dtype;

/* Shape of one prefill call. */
typedef struct kda_prefill_desc {
    int32_t num_seqs;       /* N >= 0 packed sequences */
    int32_t total_tokens;   /* T >= 0, sum of all sequence lengths */
    int32_t num_heads;      /* H >= 1 */
    int32_t dk;             /* key/query channels: 64 or 128 */
    int32_t dv;             /* value channels: must equal dk */
    int32_t qkv_dtype;      /* a kda_dtype */
    int32_t prologue;       /* KDA_PROLOGUE_* bits (0: inputs as given); others rejected */
} kda_prefill_desc;

/* Library ABI version (KDA_ABI_VERSION of the build). */
int32_t kda_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* kda_status_string(kda_status status);

/*
 * Bytes of device scratch memory kda_prefill needs for `desc` (may be 0).
 * Returns 0 for a desc that kda_prefill would reject.  Non-zero exactly when the
 * chunkwise form runs chunk-parallel: bf16, dk = dv = 128, at most 32768 (chunk, head)
 * items ((total_tokens / 64 + num_seqs) * num_heads), and a cost estimate from the shape
 * favours it over one CTA per (sequence, head): few units (up to ~130 for 8192-token
 * sequences), or a partial second wave on the 152 SMs.  The workspace then holds
 * the chunk offsets and, per (64-token chunk, head), the operands of that chunk's state
 * step: 115,200 bytes each, for (total_tokens / 64 + num_seqs) * num_heads chunks.
 */
size_t kda_prefill_workspace_bytes(const kda_prefill_desc* desc);

/* What one kda_prefill call for a given desc will do (for harnesses and tracing). */
typedef struct kda_prefill_plan {
    int32_t kernel_launches;   /* kernels one call enqueues */
    int32_t tensor_cores;      /* 1: BF16 tcgen05 path; 0: fp32 CUDA-core path */
    size_t workspace_bytes;    /* same as kda_prefill_workspace_bytes(desc) */
} kda_prefill_plan;

/*
 * Fills *plan for `desc`.  Host only, no CUDA call.  KDA_ERR_INVALID_ARG or
 * KDA_ERR_UNSUPPORTED for a desc that kda_prefill would reject.
 */
kda_status kda_prefill_query(const kda_prefill_desc* desc, kda_prefill_plan* plan);

/*
 * kda_prefill -- chunkwise-parallel KDA over varlen-packed sequences
 * (llm-atlas K3_RESEARCH.md, Q07: state passed recursively between chunks,
 * parallel matrix work inside a chunk; agihunt digest: 16-token tiles).
 *
 * Layouts (T = total_tokens, H = num_heads, N = num_seqs):
 *   q, k        [T, H, dk]   qkv_dtype
 *   v           [T, H, dv]   qkv_dtype
 *   g           [T, H, dk]   fp32, natural-log decay per key channel
 *   beta        [T, H]       fp32
 *   cu_seqlens  [N + 1]      int32, cu[0] = 0, non-decreasing, cu[N] = T;
 *                            NULL = N equal sequences (T % N must be 0)
 *   init_state  [N, H, dk, dv] fp32 (row c = key channel c); NULL = zero state
 *   out         [T, H, dv]   fp32, written for every token
 *   final_state [N, H, dk, dv] fp32; NULL = not written.  May be the same
 *                            pointer as init_state (in-place chaining of calls);
 *                            any other overlap with an input is rejected.
 *   workspace   device scratch of at least kda_prefill_workspace_bytes(desc)
 *               (may be NULL when that is 0), 16-byte aligned, overlapping no
 *               input or output; its contents need no set-up and are clobbered.
 *               Two calls in flight at once need two workspaces.  With a
 *               workspace the call computes chunk offsets, then the
 *               state-independent operands of every (chunk, head) at once and
 *               the state scan, in one cooperative launch at up to 120
 *               (sequence, head) units (two launches in all) or in two
 *               separate ones above that (three in all).  Without one, one
 *               launch.  All forms give bit-identical results.
 * A cu_seqlens entry that breaks the rules above is found on the device: that
 * sequence is skipped and kda_last_device_status() returns KDA_ERR_INVALID_ARG.
 */
kda_status kda_prefill(const kda_prefill_desc* desc,
                       const void* q, const void* k, const void* v,
                       const float* g, const float* beta,
                       const int32_t* cu_seqlens,
                       const float* init_state,
                       float* out, float* final_state,
                       void* workspace, size_t workspace_bytes,
                       void* stream);

/*
 * kda_prefill_gated -- kda_prefill with the output gate (see the top): every output
 * element is written as o * sigmoid(z), z = gate[t][h][j] (llm-atlas K3_RESEARCH.md, Q08,
 * read as an elementwise sigmoid gate on the read-out channels).
 *   gate  [T, H, dv] fp32 logits, device memory, 16-byte aligned; must not overlap out,
 *         final_state or the workspace.  NULL makes the call identical to kda_prefill.
 * Everything else (layouts, workspace, paths, errors) as kda_prefill; final_state is the
 * ungated recurrence's, bit for bit.
 */
kda_status kda_prefill_gated(const kda_prefill_desc* desc,
                             const void* q, const void* k, const void* v,
                             const float* g, const float* beta, const float* gate,
                             const int32_t* cu_seqlens,
                             const float* init_state,
                             float* out, float* final_state,
                             void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * kda_prefill_checkpointed -- kda_prefill that also snapshots each sequence's state at
 * chunk-aligned positions, for resuming a later request from a cached prefix (llm-atlas
 * K3_RESEARCH.md, Q31 hybrid prefix cache with sparse KDA checkpoints and 512-token hash
 * boundaries; section 8 device layer "KDA replay input"; Lab H boundary arithmetic).
 *
 * Same arguments and rules as kda_prefill, plus:
 *   checkpoint_interval  tokens between snapshots: a positive multiple of 64
 *   checkpoint_slots     snapshots kept per sequence (>= 1)
 *   checkpoints          [N, H, checkpoint_slots, dk, dv] fp32, device memory; slot j of
 *                        sequence n receives the state after its first (j + 1) *
 *                        checkpoint_interval tokens, for every such boundary that lies
 *                        within the sequence (the state after the whole sequence is
 *                        final_state).  Slots past a sequence's last boundary are not
 *                        written.  Must not overlap any other argument.
 * Resuming from slot j = running kda_prefill on the tokens after that boundary with
 * init_state = the snapshot.
 */
kda_status kda_prefill_checkpointed(const kda_prefill_desc* desc,
                                    const void* q, const void* k, const void* v,
                                    const float* g, const float* beta,
                                    const int32_t* cu_seqlens,
                                    const float* init_state,
                                    float* out, float* final_state,
                                    int32_t checkpoint_interval, int32_t checkpoint_slots,
                                    float* checkpoints,
                                    void* workspace, size_t workspace_bytes,
                                    void* stream);

/*
 * kda_prefill_host -- kda_prefill with q, k, v, g, beta, cu_seqlens, init_state, out and
 * final_state in HOST memory (same layouts and rules as kda_prefill; the chunkwise form
 * is the one of llm-atlas K3_RESEARCH.md, Q07).  The call walks the sequences in rounds of
 * `segment_tokens` tokens per sequence and keeps the state on the device between rounds:
 * round r's inputs are copied into one of two device staging sets on an upload stream
 * while round r-1 runs on `stream`, and round r-1's outputs are copied back on a
 * download stream (streams and events of the library, ordered after prior work on
 * `stream`).  segment_tokens is a positive multiple of 64, so the chunk boundaries, and
 * every output and final-state value, equal those of one kda_prefill call.
 *
 *   workspace   DEVICE memory of at least kda_prefill_host_workspace_bytes(desc,
 *               segment_tokens) bytes, 256-byte aligned; clobbered.
 *   stream      compute stream; when the call returns, `stream` has been made to wait for
 *               all of its copies and kernels: synchronise it before reading out or
 *               final_state, or reusing the host inputs.
 * Host buffers should be pinned (cudaHostAlloc / cudaHostRegister) for the copies to
 * overlap the kernels; pageable memory gives the same results more slowly.  Calls on one
 * device are serialised by the library while they enqueue.
 * Errors: as kda_prefill (cu_seqlens is checked on the host); KDA_ERR_INVALID_ARG for a
 * segment_tokens that is not a positive multiple of 64 or a misaligned workspace;
 * KDA_ERR_WORKSPACE for a short one.  Nothing is enqueued when an argument is rejected.  When
 * a CUDA call fails after work has been enqueued, the error is returned with `stream` made to
 * wait (as far as the runtime still allows) for the copies and kernels already enqueued, so
 * that synchronising it still marks the point after which no copy touches the buffers.
 */
size_t kda_prefill_host_workspace_bytes(const kda_prefill_desc* desc, int32_t segment_tokens);

kda_status kda_prefill_host(const kda_prefill_desc* desc,
                            const void* q, const void* k, const void* v,
                            const float* g, const float* beta,
                            const int32_t* cu_seqlens,
                            const float* init_state,
                            float* out, float* final_state,
                            int32_t segment_tokens,
                            void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * kda_prefill_host_static -- kda_prefill_host without a caller workspace.  The pages have
 * no counterpart to this entry point.  It is for callers that cannot call cudaMalloc when
 * a request arrives: a serving process that has already handed all of the device's memory
 * to its own pool (a fresh cudaMalloc would fail or fragment it), or a latency-bound loop
 * that cannot take the device-wide synchronisation a cudaMalloc may cause, and has no
 * device buffer of its own to lend.  The device staging then lives in a fixed scratch
 * array inside the library, KDA_STATIC_SCRATCH_BYTES per device, which every device that
 * loads the library holds until the process exits; the call itself calls no cudaMalloc,
 * cudaFree or allocating library routine.  Same arguments, layouts, results and stream
 * semantics as kda_prefill_host.
 *   - The first call on a device sets that device up (the scratch's device address, taken
 *     with cudaGetSymbolAddress while that device is current, and one event); make that
 *     first call before any stream capture.
 *   - Every call on a device shares the one array, which keeps whatever the last call left
 *     in it; each call writes every part of it that it reads (the state is copied in or
 *     zeroed first).  Two calls that ran on the GPU at the same time would race on it, so
 *     the library orders them: each call's copies and kernels run after those of the
 *     previous call on that device, whatever streams they were given.
 * Errors: as kda_prefill_host, and KDA_ERR_WORKSPACE when
 * kda_prefill_host_workspace_bytes(desc, segment_tokens) exceeds the scratch (a smaller
 * segment_tokens, or kda_prefill_host with a workspace, serves larger problems); nothing
 * is enqueued then.
 */
#define KDA_STATIC_SCRATCH_BYTES (64u << 20)

kda_status kda_prefill_host_static(const kda_prefill_desc* desc,
                                   const void* q, const void* k, const void* v,
                                   const float* g, const float* beta,
                                   const int32_t* cu_seqlens,
                                   const float* init_state,
                                   float* out, float* final_state,
                                   int32_t segment_tokens,
                                   void* stream);

/*
 * kda_decode -- one token per sequence, as a fused O(1) update of each head's
 * state: a single read and a single write of S (llm-atlas K3_RESEARCH.md, Q07
 * "decode keeps the O(1) state update"; section 8 device layer "fused decode").
 *
 * Layouts (B = batch):
 *   q, k   [B, H, dk]  qkv_dtype;     v [B, H, dv] qkv_dtype
 *   g      [B, H, dk]  fp32;          beta [B, H] fp32
 *   state  [B, H, dk, dv] fp32, read and overwritten in place
 *   out    [B, H, dv] fp32 (o = S_new^T q); must not overlap any input or state
 *   prologue  KDA_PROLOGUE_* bits applied to this token's inputs (see the top)
 */
kda_status kda_decode(int32_t batch, int32_t num_heads, int32_t dk, int32_t dv, int32_t qkv_dtype,
                      int32_t prologue,
                      const void* q, const void* k, const void* v,
                      const float* g, const float* beta,
                      float* state, float* out,
                      void* stream);

/*
 * kda_decode_gated -- kda_decode with the output gate: out = o * sigmoid(gate) elementwise
 * (llm-atlas K3_RESEARCH.md, Q08; see the top).  gate [B, H, dv] fp32 logits, device memory,
 * 16-byte aligned, overlapping neither out nor state; NULL = kda_decode.  The state update
 * is that of kda_decode, bit for bit.
 */
kda_status kda_decode_gated(int32_t batch, int32_t num_heads, int32_t dk, int32_t dv, int32_t qkv_dtype,
                            int32_t prologue,
                            const void* q, const void* k, const void* v,
                            const float* g, const float* beta, const float* gate,
                            float* state, float* out,
                            void* stream);

/*
 * kda_decode_multi -- K consecutive tokens of each sequence in one pass over each head's
 * state, for verifying K draft tokens (llm-atlas K3_RESEARCH.md, Q28: the MTP layer tuned
 * into an EAGLE-3 draft; Q07: O(1) decode update).  Per token the same fused update as
 * kda_decode; the state stays in registers across the K tokens, so HBM sees one read of
 * S and at most one write.
 *
 * Layouts (B = batch, K = tokens, 1 <= K <= KDA_DECODE_MULTI_MAX_TOKENS):
 *   q, k     [B, K, H, dk] qkv_dtype;   v [B, K, H, dv] qkv_dtype
 *   g        [B, K, H, dk] fp32;        beta [B, K, H] fp32
 *   n_apply  [B] int32 device memory, or NULL (= K for every sequence): the state of
 *            sequence b is replaced by the state after its first n_apply[b] tokens
 *            (0 leaves it untouched).  A value outside [0, K] leaves that state untouched
 *            and makes kda_last_device_status() return KDA_ERR_INVALID_ARG.
 *   state    [B, H, dk, dv] fp32, read, and written where n_apply[b] > 0
 *   out      [B, K, H, dv] fp32, o for every token (whatever n_apply says), or NULL
 * Verification: one call with n_apply = 0 (outputs for all K drafts, state untouched),
 * then one with n_apply = the accepted count per sequence and out = NULL.
 * prologue: KDA_PROLOGUE_* bits applied to every token's inputs (see the top).
 * Errors: as kda_decode, plus KDA_ERR_INVALID_ARG for K out of range.
 */
#define KDA_DECODE_MULTI_MAX_TOKENS 64

kda_status kda_decode_multi(int32_t batch, int32_t tokens, int32_t num_heads, int32_t dk, int32_t dv,
                            int32_t qkv_dtype, int32_t prologue,
                            const void* q, const void* k, const void* v,
                            const float* g, const float* beta,
                            const int32_t* n_apply,
                            float* state, float* out,
                            void* stream);

/*
 * kda_decode_multi_gated -- kda_decode_multi with the output gate on every token's output:
 * out = o * sigmoid(gate) (llm-atlas K3_RESEARCH.md, Q08; see the top).  gate [B, K, H, dv]
 * fp32 logits, device memory, 16-byte aligned, overlapping neither out nor state; ignored
 * when out is NULL; NULL = kda_decode_multi.  States as kda_decode_multi, bit for bit.
 */
kda_status kda_decode_multi_gated(int32_t batch, int32_t tokens, int32_t num_heads, int32_t dk, int32_t dv,
                                  int32_t qkv_dtype, int32_t prologue,
                                  const void* q, const void* k, const void* v,
                                  const float* g, const float* beta, const float* gate,
                                  const int32_t* n_apply,
                                  float* state, float* out,
                                  void* stream);

/*
 * kda_state_combine -- the fold step of context-parallel prefill over one long sequence
 * (llm-atlas K3_RESEARCH.md, section 8 system-state table: "KCP" in the pretraining row; Q07:
 * the state passed from chunk to chunk).  When consecutive token ranges of a sequence run on
 * different ranks, range r maps the state entering it as S_after = M_r S_before + S_r, where
 * M_r is the dk x dk product of its chunks' transitions (the state after the range from
 * initial state I with v = 0: kda_prefill with a zero v and an identity init_state) and S_r
 * is the state after the range from a zero start.  The state entering range r is then the
 * fold S <- M_j S + S_j over the ranges j < r, one call per step:
 *
 *   state_out[i] = transition[i] . state_in[i] + state_add[i]     for i < count (fp32)
 *
 *   count       number of (sequence, head) states, >= 0
 *   dk, dv      must be equal, 64 or 128 (else KDA_ERR_UNSUPPORTED)
 *   transition  [count, dk, dk] fp32, row-major (may be NULL when state_in is NULL)
 *   state_in    [count, dk, dv] fp32, row c = key channel c; NULL = zero
 *   state_add   [count, dk, dv] fp32; NULL = zero
 *   state_out   [count, dk, dv] fp32; may be state_add itself (in place), must not overlap
 *               state_in or transition (KDA_ERR_INVALID_ARG)
 * All pointers are device memory, 16-byte aligned; asynchronous on `stream`.
 */
kda_status kda_state_combine(int32_t count, int32_t dk, int32_t dv,
                             const float* transition, const float* state_in,
                             const float* state_add, float* state_out,
                             void* stream);

/*
 * Synchronises `stream`, then returns and clears the device status word of the
 * current device: KDA_OK, KDA_ERR_INVALID_ARG (bad cu_seqlens seen on the
 * device) or KDA_ERR_TIMEOUT (a bounded wait gave up).  KDA_ERR_CUDA if the
 * synchronisation itself fails.
 */
kda_status kda_last_device_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
