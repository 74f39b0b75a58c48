// Internal launchers of the KDA library (host side).  Not part of the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kda {

struct PrefillArgs {
    int num_seqs, total_tokens, num_heads, dk, dv;
    bool bf16;
    const void *q, *k, *v;
    const float *g, *beta;
    const int32_t* cu_seqlens;
    const float* init_state;
    float *out, *final_state;
    // optional state snapshots: every ckpt_interval tokens (multiple of 64) of each
    // sequence, up to ckpt_slots per sequence, into checkpoints [N, H, ckpt_slots, dk, dv]
    int ckpt_interval, ckpt_slots;
    float* checkpoints;
    void* workspace;
    size_t workspace_bytes;
    int* status;  // device status word
    int prologue; // KDA_PROLOGUE_* bits
    const float* gate;  // output gate logits [T, H, dv] (out = o * sigmoid(gate)), or nullptr
};

struct DecodeArgs {
    int batch, num_heads, dk, dv;
    bool bf16;
    const void *q, *k, *v;
    const float *g, *beta;
    float *state, *out;
    int prologue; // KDA_PROLOGUE_* bits
    const float* gate;  // output gate logits [B, H, dv], or nullptr
};

struct DecodeMultiArgs {
    int batch, tokens, num_heads, dk, dv;
    bool bf16;
    const void *q, *k, *v;       // [B, K, H, d]
    const float *g, *beta;       // [B, K, H, dk], [B, K, H]
    const int32_t* n_apply;      // [B] tokens whose update is kept, or nullptr (= K)
    float *state, *out;          // [B, H, dk, dv] in place; [B, K, H, dv] or nullptr
    int* status;                 // device status word
    int prologue;                // KDA_PROLOGUE_* bits
    const float* gate;           // output gate logits [B, K, H, dv], or nullptr
};

// fp32 CUDA-core chunkwise prefill (any supported shape, fp32 or bf16 inputs)
cudaError_t launch_prefill_simt(const PrefillArgs& a, cudaStream_t stream);
// bf16 tcgen05 chunkwise prefill (dk = dv = 128, T > 0)
cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t stream);
// the same, chunk-parallel: per-chunk operands for every chunk at once (workspace), then
// the state scan; needs prefill_split_workspace_bytes of workspace, 16-byte aligned
cudaError_t launch_prefill_split(const PrefillArgs& a, cudaStream_t stream);
size_t prefill_split_workspace_bytes(int num_seqs, int total_tokens, int num_heads);
// fused single-pass decode
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
// K tokens per sequence in one pass over the state
cudaError_t launch_decode_multi(const DecodeMultiArgs& a, cudaStream_t stream);

}  // namespace kda
