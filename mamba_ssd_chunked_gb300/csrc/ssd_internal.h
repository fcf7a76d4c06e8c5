// Host-side declarations shared by the translation units of libssd.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "ssd.h"

namespace ssd {

// One forward call, arguments already validated.
struct FwdArgs {
    ssd_dims d;
    ssd_dtype io;
    const void* x;
    const float* dt;
    const float* dt_bias;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const float* init;
    int chunk_len;
    void* y;
    float* final_state;
    cudaStream_t stream;
    unsigned* status_word;             // device word: bit 0 = a bounded wait timed out
    unsigned long long wait_limit_ns;  // per-wait wall-clock limit on the device
    float dt_min = 0.f;                // softplus(dt + dt_bias) is clamped to [dt_min, dt_max]
    float dt_max = __builtin_inff();
    // chain path: where a chain crosses into this CTA, recompute its state over the
    // blocks it takes to decay away instead of waiting for the previous CTA's hand-off:
    // 0 never, 1 when the hand-off would come late, 2 whenever possible
    int chain_warmup = 1;
    // [batch, seqlen] packed-sequence ids (nullable): the state restarts from
    // zero wherever the id changes between consecutive tokens of a row
    const int32_t* seq_idx = nullptr;
};

// A change of seq_idx before token t adds -kSeqCutNats to that token's
// log-decay dt*A in every path's cumulative sum. The state carried across is
// then scaled by e^{-256 + at most 75} (the largest positive exponent of any
// path's factored form), exactly 0 in fp32: the restart is exact, and the
// paths' large-decay handling (split blocks, per-entry masks) takes it as is.
constexpr float kSeqCutNats = 256.f;

// CUDA-core path: the five stages at exactly chunk_len, chunk states in workspace.
bool simt_supported(const ssd_dims& d, int chunk_len);
size_t simt_workspace_bytes(const ssd_dims& d, int chunk_len);
ssd_status simt_forward(const FwdArgs& a, void* ws, size_t ws_bytes);

// Fused tcgen05/TMA path.
bool tc_supported(const ssd_dims& d, ssd_dtype io, int chunk_len);
size_t tc_workspace_bytes(const ssd_dims& d, int chunk_len);
ssd_status tc_forward(const FwdArgs& a, void* ws, size_t ws_bytes);

// Chain-local fused tcgen05/TMA path (dstate 128 or 256): persistent CTAs, state kept on chip.
bool chain_supported(const ssd_dims& d, ssd_dtype io, int chunk_len);
size_t chain_workspace_bytes(const ssd_dims& d);
ssd_status chain_forward(const FwdArgs& a, void* ws, size_t ws_bytes);

// 4-D bf16 TMA map over a row-major [outer, rows, mid, inner] tensor, box
// {64, 1, box_rows, 1}, 128-byte swizzle, zero fill out of bounds.
bool make_map_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t mid, uint64_t rows, uint64_t outer,
                   uint32_t box_rows = 128);

// One decode step on a carried state (ssd_step), arguments already validated.
struct StepArgs {
    ssd_dims d;
    ssd_dtype io;
    const void* x;
    const float* dt;
    const float* dt_bias;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    float* state;
    void* y;
    cudaStream_t stream;
    float dt_min = 0.f;  // softplus(dt + dt_bias) is clamped to [dt_min, dt_max]
    float dt_max = __builtin_inff();
};
bool step_supported(const ssd_dims& d);
ssd_status step_forward(const StepArgs& a);

// The inputs of one forward for the input guard (ssd_check_inputs), already
// validated: x, B, C element-aligned in io, the fp32 ones 4-byte aligned.
struct CheckArgs {
    ssd_dims d;
    ssd_dtype io;
    const void* x;
    const float* dt;
    const float* dt_bias;
    const float* A;
    const void* B;
    const void* C;
    const float* D;     // nullable
    const float* init;  // nullable
    cudaStream_t stream;
};
// Non-finite element counts of x, dt, dt_bias, A, B, C, D, init into counts[8]
// (host); synchronizes a.stream.
ssd_status check_inputs(const CheckArgs& a, int64_t* counts);

// Launch bookkeeping (every kernel launch of the library goes through it).
void note_launches(uint64_t n);

// ssd_kernel_timing: event pair around a forward's main kernel on its stream
// (no-ops while timing is off)
void timing_begin(cudaStream_t s);
void timing_end(cudaStream_t s);

constexpr size_t kWorkspaceAlign = 256;
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace ssd
