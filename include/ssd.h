/*
 * ssd.h -- C ABI of libssd: the Mamba-2 SSD (state-space duality) chunked-scan
 * forward on one NVIDIA GB300 (sm_103a).
 *
 * The operation (the same one, whatever path computes it):
 *
 *   delta[b,t,h] = softplus(dt[b,t,h] + dt_bias[h])   (ssd_fwd_ex / ssd_step_ex: clamped, ssd_dt_limit)
 *   s_{-1}       = init_state[b,h]        (zeros when init_state == NULL)
 *   s_{t-1}      = 0 where seq_idx[b,t] != seq_idx[b,t-1], t > 0   (ssd_fwd_ex with seq_idx only)
 *   s_t          = exp(delta[b,t,h] A[h]) s_{t-1} + delta[b,t,h] x[b,t,h,:] (outer) B[b,t,g(h),:]
 *   y[b,t,h,:]   = s_t C[b,t,g(h),:] + D[h] x[b,t,h,:]           (D == NULL: no skip)
 *   final_state[b,h] = s_{L-1}
 *   g(h) = h / (nheads / ngroups)
 *
 * Sources: flash-linear-attention "fla/layers/mamba2.py" (Mamba2.torch_forward,
 * the naive chunked SSD; the mamba_chunk_scan_combined call with
 * dt_softplus=True, dt_bias, D, return_final_states=True); burn-mamba
 * "mamba2/ssd/serial.rs" (ssd_serial and kernels k1..k5: chunk cumsum of
 * dt*A, C.B^T per chunk, chunk states, serial state passing, chunk scan with
 * the exp-segsum mask and D skip); burn-mamba "Mamba2SsdInput" rustdoc
 * (ssd_minimal, Steps 1-4, paper Section 4.1 Eq. 20/22/23); lrnnx
 * "ops/selective_scan.html" (selective_scan_ref: the token recurrence).
 *
 * Layouts: every tensor is a dense, row-major (C-contiguous) array.
 *   x, y         [batch, seqlen, nheads, headdim]   io dtype (fp32 or bf16)
 *   B, C         [batch, seqlen, ngroups, dstate]   io dtype
 *   dt           [batch, seqlen, nheads]            fp32, raw (before bias and softplus)
 *   dt_bias, A, D [nheads]                          fp32; A must be < 0 for a decaying state
 *   init_state, final_state [batch, nheads, headdim, dstate]  fp32
 *
 * Ownership: the caller owns every buffer it passes. Device pointers must be
 * device-resident on the current CUDA device and 16-byte aligned. Calls are
 * asynchronous on `stream` (a cudaStream_t; NULL is the legacy default
 * stream) unless stated otherwise; the library keeps no pointer to caller
 * memory after a call returns.
 *
 * Errors: no entry point aborts, traps or throws. Arguments are checked on
 * the host before anything is launched. A device-side wait that runs past
 * its time limit records SSD_ERR_DEVICE_TIMEOUT in a per-device status word
 * (see ssd_device_status) instead of hanging.
 */
#ifndef SSD_H_
#define SSD_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SSD_API __attribute__((visibility("default")))
#else
#define SSD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARG = 1,     /* bad dims, NULL required pointer, ngroups mismatch, ... */
    SSD_ERR_UNSUPPORTED = 2,     /* valid but outside what the chosen path implements */
    SSD_ERR_CUDA = 3,            /* a CUDA runtime/driver call failed */
    SSD_ERR_DEVICE_TIMEOUT = 4,  /* a bounded device-side wait gave up */
    SSD_ERR_WORKSPACE = 5,       /* caller workspace too small or misaligned */
    SSD_ERR_DEBUG_CHECK = 6      /* debug build only: a kernel's index or bounds check failed */
} ssd_status;

typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype;

/* Which kernels compute the forward.
 *   SSD_PATH_AUTO:  SSD_PATH_CHAIN when supported, else SSD_PATH_TC when
 *                   supported, else the SIMT path.
 *   SSD_PATH_SIMT:  fp32 CUDA-core kernels, any supported shape, the five
 *                   stages at exactly chunk_len (chunk states in workspace).
 *   SSD_PATH_TC:    fused tcgen05/TMA kernel, one CTA per (128-token block,
 *                   head group), chunk states chained through workspace
 *                   (bf16 io, headdim 64, dstate 128 or 256, chunk_len 128
 *                   or 256).
 *   SSD_PATH_CHAIN: fused tcgen05/TMA kernel, one persistent CTA per SM that
 *                   walks whole chains block by block with the chunk state
 *                   kept in tensor memory (bf16 io, headdim 64 with an even
 *                   number of heads per group, or headdim 128; dstate 128 or
 *                   256; chunk_len 128 or 256). Its workspace depends on the
 *                   current device's SM count. */
typedef enum { SSD_PATH_AUTO = 0, SSD_PATH_SIMT = 1, SSD_PATH_TC = 2, SSD_PATH_CHAIN = 3 } ssd_path;

typedef struct {
    int64_t batch, seqlen, nheads, headdim, ngroups, dstate;
} ssd_dims;

/* Clamp of the discretisation step: delta = min(max(softplus(dt + dt_bias),
 * dt_min), dt_max), torch.clamp's order (fla "mamba2.py", Mamba2.torch_forward:
 * the time_step_limit clamp after softplus; the fused branch passes it as
 * dt_limit). Requires 0 <= dt_min <= dt_max; dt_max may be +INFINITY.
 * {0, INFINITY} (or a NULL pointer where one is taken) changes nothing.
 * Padded steps past the sequence end keep delta = 0. */
typedef struct {
    float dt_min, dt_max;
} ssd_dt_limit;

/*
 * ssd_fwd -- the SSD chunked-scan forward (the five stages of burn-mamba
 * "serial.rs" ssd_serial / fla "mamba2.py" naive chunked SSD).
 *
 * dims            shapes; every field >= 1; nheads % ngroups == 0.
 * io_dtype        dtype of x, B, C and y.
 * x, dt, dt_bias, A, B, C   device inputs (required).
 * D               device [nheads] fp32 or NULL (no skip term).
 * init_state      device [b,h,p,n] fp32 or NULL (zero initial state).
 * chunk_len       chunk length Q, 1..256 (SIMT); 128 or 256 (tensor-core path).
 * ngroups         must equal dims->ngroups.
 * y               device output [b,L,h,p], io dtype (required).
 * final_state     device output [b,h,p,n] fp32, or NULL (not written).
 * stream          cudaStream_t.
 *
 * Scratch comes from a library-owned per-device workspace that grows on
 * demand (cudaMalloc on first use or growth; freed by ssd_release). Calls
 * that share that workspace must not overlap on the device: issue them on
 * one stream, or use ssd_fwd_ws with a workspace per stream.
 * Returns SSD_OK once the work is enqueued.
 */
SSD_API ssd_status ssd_fwd(const ssd_dims* dims, ssd_dtype io_dtype,
                   const void* x, const float* dt, const float* dt_bias, const float* A,
                   const void* B, const void* C, const float* D, const float* init_state,
                   int chunk_len, int ngroups, void* y, float* final_state, void* stream);

/*
 * ssd_fwd_ws -- ssd_fwd with an explicit path and caller-owned device
 * workspace of at least ssd_fwd_workspace_bytes(...) bytes, 256-byte aligned.
 * Zero-fill the workspace once before its first use and keep it for this
 * library afterwards: the tensor-core path passes chunk states between CTAs
 * through it as tagged words, and a tag is only trusted because stale
 * contents can only be zeros or this library's own earlier tags. The
 * workspace must not be used by another call that overlaps on the device.
 */
SSD_API ssd_status ssd_fwd_ws(const ssd_dims* dims, ssd_dtype io_dtype,
                      const void* x, const float* dt, const float* dt_bias, const float* A,
                      const void* B, const void* C, const float* D, const float* init_state,
                      int chunk_len, int ngroups, void* y, float* final_state,
                      ssd_path path, void* workspace, size_t workspace_bytes, void* stream);

/*
 * ssd_fwd_ex -- ssd_fwd with a dt limit, packed sequences, and an optional
 * explicit path and workspace (fla "fla/layers/mamba2.py": the dt_limit and
 * seq_idx arguments of the fused chunked-scan call).
 *
 * dt_limit        NULL: no clamp; else delta = min(max(softplus(..), dt_min), dt_max)
 *                 (SSD_ERR_INVALID_ARG when dt_min < 0, dt_max < dt_min or either is NaN).
 * seq_idx         NULL, or device [batch, seqlen] int32 (4-byte aligned; else
 *                 SSD_ERR_UNSUPPORTED): several sequences packed into each row.
 *                 Wherever seq_idx changes between consecutive tokens of a row
 *                 the state restarts from zero (no state crosses; any int32
 *                 values, increasing or not). init_state is the state before
 *                 the row's first token and final_state the state after its
 *                 last. The pages pass seq_idx but do not define it further;
 *                 this is the reading taken.
 * workspace       NULL: the library-owned workspace (as ssd_fwd, path
 *                 honoured); else a caller workspace under the rules of ssd_fwd_ws.
 * Everything else as ssd_fwd.
 */
SSD_API ssd_status ssd_fwd_ex(const ssd_dims* dims, ssd_dtype io_dtype,
                              const void* x, const float* dt, const float* dt_bias, const float* A,
                              const void* B, const void* C, const float* D, const float* init_state,
                              int chunk_len, int ngroups, void* y, float* final_state,
                              const ssd_dt_limit* dt_limit, const int32_t* seq_idx, ssd_path path,
                              void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes ssd_fwd_ws needs for these arguments (0 if they are invalid). */
SSD_API size_t ssd_fwd_workspace_bytes(const ssd_dims* dims, ssd_dtype io_dtype, int chunk_len, ssd_path path);

/* The path SSD_PATH_AUTO picks for these arguments (never SSD_PATH_AUTO). */
SSD_API ssd_path ssd_select_path(const ssd_dims* dims, ssd_dtype io_dtype, int chunk_len);

/*
 * ssd_fwd_host -- end-to-end call on HOST buffers (same layouts and meaning
 * as ssd_fwd; pinned host memory makes the copies asynchronous). Copies the
 * inputs to library-owned device buffers, runs the forward, copies y (and
 * final_state when non-NULL) back, and synchronizes `stream` before
 * returning, so the outputs are ready on return. The sequence is cut into
 * token slices, each covering every batch row: one per 96 MiB of copies, at
 * least 4 and at most 16, none shorter than 512 tokens, cuts on multiples of
 * 256 (the environment variable SSD_HOST_SLICES, 1 to 16, replaces the count
 * from the copies). A slice's final state is the next slice's initial state,
 * which is exact for any cut (results match one ssd_fwd call up to rounding). Library-owned streams upload, compute and download the slices
 * in order, so that one slice's upload overlaps another's forward and a third's
 * download; they start after the work already queued on `stream`, which waits
 * for all of them before the call returns. Device-side timeouts are reported
 * in the return value. The staging buffers and streams belong to the device:
 * ssd_fwd_host calls on one device must not overlap (issue them from one host
 * thread at a time).
 */
SSD_API ssd_status ssd_fwd_host(const ssd_dims* dims, ssd_dtype io_dtype,
                        const void* x, const float* dt, const float* dt_bias, const float* A,
                        const void* B, const void* C, const float* D, const float* init_state,
                        int chunk_len, int ngroups, void* y, float* final_state, void* stream);

/* The number of token slices ssd_fwd_host cuts a call with these dims into
 * (after SSD_HOST_SLICES, if set); 0 for invalid dims. Host only. */
SSD_API int ssd_host_slices(const ssd_dims* dims, ssd_dtype io_dtype);

/*
 * ssd_check_inputs -- the input guard: counts the non-finite elements (NaN,
 * +Inf, -Inf) of each input of an ssd_fwd call with these dims. The burn-mamba
 * port runs a sanity check on every input before its kernels (`mamba2/ssd/
 * serial.rs`, Mamba2::ssd_serial: x, dt, A, B, C, D and the initial state);
 * a non-finite input spreads through the state to every later token of its
 * chain, so a caller may refuse the forward instead.
 *   dims, io_dtype, x, dt, dt_bias, A, B, C, D, init_state: as for ssd_fwd
 *                 (device pointers, contiguous; x, B, C in io_dtype, the rest
 *                 fp32; D and init_state may be NULL). Each pointer needs only
 *                 its element's alignment. The inputs are only read.
 *   counts        host int64[8], written on success: the counts for x, dt,
 *                 dt_bias, A, B, C, D, init_state in that order (0 for a NULL
 *                 D or init_state).
 * One kernel over the eight tensors on `stream` (HBM bound: one read of each);
 * the call synchronizes `stream` to return the counts. Errors:
 * SSD_ERR_INVALID_ARG (NULL dims, counts or required input; dims < 1;
 * nheads % ngroups != 0; unknown dtype), SSD_ERR_UNSUPPORTED (a pointer not
 * aligned to its element), SSD_ERR_CUDA.
 */
SSD_API ssd_status ssd_check_inputs(const ssd_dims* dims, ssd_dtype io_dtype,
                        const void* x, const float* dt, const float* dt_bias, const float* A,
                        const void* B, const void* C, const float* D, const float* init_state,
                        int64_t* counts, void* stream);

/* Synchronizes `stream`, then returns and clears the current device's status
 * word: SSD_OK, SSD_ERR_DEVICE_TIMEOUT, SSD_ERR_DEBUG_CHECK (debug build only,
 * see ssd_debug_build), or SSD_ERR_CUDA if the sync failed. */
SSD_API ssd_status ssd_device_status(void* stream);

/*
 * Debug build (libssd_debug.so, compiled with SSD_DEBUG; the stand-in for a
 * memory checker): every index the tensor-core kernels compute by hand (ring,
 * X/W and table slots, tensor-memory columns, TMA coordinates, global state
 * rows, job positions) is checked before use. A failed check skips that
 * access (a skipped copy then ends in a bounded-wait timeout, never in a
 * fault), and ssd_device_status reports SSD_ERR_DEBUG_CHECK.
 * ssd_debug_build: 1 in that build, 0 in the release build.
 * ssd_debug_failed_line: source line of the first failed check since the last
 * ssd_device_status call that saw it (0: none; always 0 in the release build);
 * call it before ssd_device_status, which clears it. Synchronizes `stream`.
 */
SSD_API int ssd_debug_build(void);
SSD_API unsigned ssd_debug_failed_line(void* stream);

/* Static, human-readable name of a status code. */
SSD_API const char* ssd_status_string(ssd_status status);

/* Kernels this library has launched in this process (all devices, all calls). */
SSD_API uint64_t ssd_kernel_launches(void);

/*
 * Device time of each forward's fused kernel, for measurement. While enabled
 * (enable != 0), every ssd_fwd* call records a CUDA event pair on its stream
 * right before and after the launch of its main kernel (the fused kernel of
 * the tensor-core paths, the three kernels of the SIMT path). An event record
 * between launches keeps consecutive kernels from overlapping, so enable it
 * only for a measurement pass. ssd_kernel_timing_read waits for the recorded
 * pairs (all of the current device), writes their summed elapsed time in
 * milliseconds and their number, and forgets them. Returns SSD_ERR_INVALID_ARG
 * for NULL outputs and SSD_ERR_CUDA if a CUDA event call failed.
 */
SSD_API void ssd_kernel_timing(int enable);
SSD_API ssd_status ssd_kernel_timing_read(double* total_ms, uint64_t* count);

/* Frees the library-owned device and pinned buffers of every device. Not safe
 * while calls that use them are in flight. */
SSD_API void ssd_release(void);

/*
 * ssd_fwd_noalloc -- the fused tensor-core forward on a fixed scratch array
 * compiled into the library, for callers that must not allocate device
 * memory: code running under a memory manager that owns all of the device's
 * memory and forbids allocations behind its back, and latency-critical loops
 * where cudaMalloc (which may synchronise the device) is not acceptable. (The
 * pages have no counterpart: their kernels allocate their intermediates.)
 *
 * Arguments, layouts and results are those of ssd_fwd; the inputs and outputs
 * are still the caller's buffers. Only the tensor-core path runs here
 * (SSD_ERR_UNSUPPORTED otherwise). The scratch is a 16 MiB (16777216-byte)
 * file-scope device array; a call whose scratch need (ssd_fwd_workspace_bytes
 * with SSD_PATH_TC) exceeds it returns SSD_ERR_WORKSPACE before launching
 * anything: at most 255 (batch, head) chains at dstate 128, 127 at dstate 256.
 *
 * No cudaMalloc, cudaFree or allocating library routine is called. The first
 * call on a device looks up the array's device address and zero-fills it,
 * synchronously, so make that first call before any stream capture. Every call
 * on a device shares the one array and it keeps the last call's contents (the
 * per-call work counter is cleared by each call): calls that overlap on the
 * GPU, on any streams, race and must not be issued.
 */
SSD_API ssd_status ssd_fwd_noalloc(const ssd_dims* dims, ssd_dtype io_dtype,
                                   const void* x, const float* dt, const float* dt_bias, const float* A,
                                   const void* B, const void* C, const float* D, const float* init_state,
                                   int chunk_len, int ngroups, void* y, float* final_state, void* stream);

/*
 * ssd_step -- one decode step: a single new token per sequence, applied to a
 * carried SSM state (fla "mamba2.py", Mamba2.torch_forward, cached-decode
 * branch; its fast path is selective_state_update):
 *
 *   dt'  = softplus(dt + dt_bias[h])
 *   state[b,h,p,n] = exp(dt' A[h]) state[b,h,p,n] + dt' x[b,h,p] B[b,g,n]
 *   y[b,h,p]       = sum_n state[b,h,p,n] C[b,g,n] + D[h] x[b,h,p]
 *
 * with g = h / (nheads / ngroups), the same step as ssd_fwd over one token.
 * dims->seqlen must be 1 (SSD_ERR_INVALID_ARG otherwise); the other dims are
 * those of ssd_fwd. Layouts (dense, row-major, device pointers): x and y
 * [b, h, p] in io_dtype; dt [b, h] fp32 (before bias and softplus); B and C
 * [b, g, n] in io_dtype; dt_bias, A, D [h] fp32 (D nullable); state
 * [b, h, p, n] fp32, read and overwritten in place (required). Pointers must
 * be 16-byte aligned (SSD_ERR_UNSUPPORTED). The caller owns every buffer; the
 * call is asynchronous on `stream` and needs no workspace. Arguments are
 * checked on the host before anything is launched.
 */
SSD_API ssd_status ssd_step(const ssd_dims* dims, ssd_dtype io_dtype,
                            const void* x, const float* dt, const float* dt_bias, const float* A,
                            const void* B, const void* C, const float* D, float* state,
                            int ngroups, void* y, void* stream);

/* ssd_step_ex -- ssd_step with a dt limit (NULL: none; see ssd_dt_limit). */
SSD_API ssd_status ssd_step_ex(const ssd_dims* dims, ssd_dtype io_dtype,
                               const void* x, const float* dt, const float* dt_bias, const float* A,
                               const void* B, const void* C, const float* D, float* state,
                               int ngroups, void* y, const ssd_dt_limit* dt_limit, void* stream);

/* ------------------------------------------------------------------------
 * The per-token operations around the scan in a Mamba-2 layer (fla
 * "mamba2.py", Mamba2.torch_forward, steps 2 and 3). They read and write
 * each element once: HBM-bound streaming kernels, fp32 arithmetic.
 */

/* Shapes of the conv over xBC: conv_dim = d_inner + 2 * ngroups * dstate
 * channels per token (x first, then B, then C), kernel_size taps (1..8). */
typedef struct {
    int64_t batch, seqlen, d_inner, ngroups, dstate, kernel_size;
} ssd_conv_dims;

/*
 * ssd_conv1d_silu -- causal depthwise conv1d over time plus SiLU, split into
 * the scan's inputs (fla "mamba2.py": Mamba2.__init__ builds
 * nn.Conv1d(conv_dim, conv_dim, kernel_size, groups=conv_dim,
 * padding=kernel_size - 1); Mamba2.torch_forward step 2 keeps the first
 * seqlen outputs, applies SiLU and splits x / B / C):
 *
 *   o[b,t,c] = bias[c] + sum_{k<K} weight[c,k] * xbc[b, t-(K-1)+k, c]   (zero before t = 0)
 *   x[b,t,:] = act(o[b,t,0:d_inner]); B[b,t,:] = act(o[b,t,d_inner:d_inner+G]);
 *   C[b,t,:] = act(o[b,t,d_inner+G:]),  G = ngroups*dstate, act = SiLU or identity
 *
 * xbc             device [batch, seqlen, *] io dtype; token t of sequence b
 *                 starts at xbc + (b*seqlen + t) * xbc_row_stride elements
 *                 (xbc_row_stride >= conv_dim, e.g. the in_proj row length,
 *                 so the slice can be read in place).
 * weight          device [conv_dim, kernel_size] fp32; bias [conv_dim] fp32 or NULL.
 * activation      1: SiLU; 0: none.
 * x, B, C         device outputs, dense: x [batch, seqlen, d_inner] (the
 *                 scan's [b, L, h, p]), B and C [batch, seqlen, ngroups, dstate].
 * conv_state      device output [batch, conv_dim, kernel_size] io dtype, or
 *                 NULL: the last kernel_size inputs of each channel, zeros
 *                 in front when seqlen < kernel_size (what the layer caches).
 * Pointers need the element alignment; 16-byte aligned pointers and strides
 * with d_inner, G multiples of 8 (bf16) / 4 (fp32) take the vector path.
 * Errors: SSD_ERR_INVALID_ARG (NULL, dims < 1, stride < conv_dim),
 * SSD_ERR_UNSUPPORTED (kernel_size > 8, misaligned pointer, sizes beyond the
 * indexing limits). Asynchronous on `stream`; no workspace.
 */
SSD_API ssd_status ssd_conv1d_silu(const ssd_conv_dims* dims, ssd_dtype io_dtype,
                                   const void* xbc, int64_t xbc_row_stride,
                                   const float* weight, const float* bias, int activation,
                                   void* x, void* B, void* C, void* conv_state, void* stream);

/*
 * ssd_conv1d_step -- the cached-decode form of the same conv (fla
 * "mamba2.py", Mamba2.torch_forward step 2, cache_position > 0): per
 * sequence the conv state shifts left by one token, the new token enters at
 * the right, and o[c] = bias[c] + sum_k state[c,k] * weight[c,k].
 * dims->seqlen must be 1. xbc: [batch, *] with row stride xbc_row_stride;
 * conv_state [batch, conv_dim, kernel_size] io dtype, updated in place
 * (required); x [batch, d_inner], B and C [batch, ngroups*dstate].
 * Errors and alignment as ssd_conv1d_silu.
 */
SSD_API ssd_status ssd_conv1d_step(const ssd_conv_dims* dims, ssd_dtype io_dtype,
                                   const void* xbc, int64_t xbc_row_stride,
                                   const float* weight, const float* bias, int activation,
                                   void* conv_state, void* x, void* B, void* C, void* stream);

/*
 * ssd_gated_rmsnorm -- RMSNormGated(dim, eps, norm_before_gate=False) applied
 * as norm(y, z) after the scan (fla "mamba2.py", step 3): per row and per
 * group of group_size consecutive channels,
 *
 *   v = y * silu(z)          (v = y when z == NULL)
 *   out = v / sqrt(mean(v^2 over the group) + eps) * weight
 *
 * y, z, out       device [rows, *] io dtype with the given row strides
 *                 (elements, >= dim); z may be NULL.
 * weight          device [dim] fp32.
 * group_size      channels per normalisation group; <= 0 means dim (one
 *                 group); dim % group_size == 0; at most 64 groups.
 * Errors: SSD_ERR_INVALID_ARG (NULL, sizes < 1, strides < dim, dim not a
 * multiple of group_size, eps < 0), SSD_ERR_UNSUPPORTED (more than 64
 * groups, misaligned pointers, sizes beyond the indexing limits).
 * Asynchronous on `stream`; no workspace.
 */
SSD_API ssd_status ssd_gated_rmsnorm(ssd_dtype io_dtype, int64_t rows, int64_t dim, int64_t group_size,
                                     const void* y, int64_t y_row_stride, const void* z, int64_t z_row_stride,
                                     const float* weight, float eps, void* out, int64_t out_row_stride,
                                     void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SSD_H_ */
