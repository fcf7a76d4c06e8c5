// CUDA-core (SIMT) path of the SSD forward: the five stages of the chunked
// decomposition at exactly the caller's chunk_len, in fp32 arithmetic, for
// fp32 or bf16 io. It serves fp32 inputs (where a 1e-4 relative bound rules
// out bf16 tensor-core operands) and any shape the tensor-core kernel does
// not cover.
//
// Stages (burn-mamba "mamba2/ssd/serial.rs", ssd_serial; fla "mamba2.py",
// Mamba2.torch_forward naive chunked SSD):
//   k1 chunk cumsum of dt*A  -> recomputed inside simt_chunk_state and simt_chunk_scan
//   k3 chunk states          -> simt_chunk_state (states[b,c,h,p,n], chunk log-decay)
//   k4 state passing         -> simt_state_pass (overwrites states with each chunk's input state)
//   k2 C.B^T and k5 scan     -> simt_chunk_scan (per 32-row tile of a chunk)
#include <cuda_bf16.h>

#include <algorithm>

#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxChunk = 256;
constexpr int kRows = 32;        // rows (tokens) staged per tile
constexpr int kAcc = 32;         // accumulators per thread in simt_chunk_state

template <typename T>
__device__ __forceinline__ float load_f(const T* p);
template <>
__device__ __forceinline__ float load_f<float>(const float* p) {
    return *p;
}
template <>
__device__ __forceinline__ float load_f<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}

template <typename T>
__device__ __forceinline__ void store_f(T* p, float v);
template <>
__device__ __forceinline__ void store_f<float>(float* p, float v) {
    *p = v;
}
template <>
__device__ __forceinline__ void store_f<__nv_bfloat16>(__nv_bfloat16* p, float v) {
    *p = __float2bfloat16_rn(v);
}

// softplus(v) = log(1 + e^v), evaluated without overflow.
__device__ __forceinline__ float softplus_f(float v) {
    return v > 0.f ? v + log1pf(expf(-v)) : log1pf(expf(v));
}

// k1 for chunk c of chain (b, h): s_dt[t] = softplus(dt + dt_bias) clamped to
// [lim.x, lim.y] (0 past the sequence end: padding comes after discretisation), s_cs[t] = inclusive
// cumulative sum of dt*A within the chunk, with -kSeqCutNats at each token
// where seq_idx (if given) changes. Needs blockDim.x == 256, Q <= 256.
__device__ void chunk_dt_cumsum(const float* __restrict__ dt, const float* __restrict__ dt_bias,
                                const float* __restrict__ A, const int32_t* __restrict__ seq, int64_t b, int h,
                                int c, int Q, int64_t L, int H, float2 lim, float* s_dt, float* s_cs,
                                float* s_warp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t t = static_cast<int64_t>(c) * Q + tid;
    float dtv = 0.f;
    if (tid < Q && t < L) dtv = fminf(fmaxf(softplus_f(dt[(b * L + t) * H + h] + dt_bias[h]), lim.x), lim.y);
    float v = dtv * A[h];
    if (seq && tid < Q && t > 0 && t < L && seq[b * L + t] != seq[b * L + t - 1]) v -= kSeqCutNats;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
    }
    if (lane == 31) s_warp[warp] = v;
    __syncthreads();
    float pre = 0.f;
    for (int w = 0; w < warp; ++w) pre += s_warp[w];
    if (tid < Q) {
        s_dt[tid] = dtv;
        s_cs[tid] = v + pre;
    }
    __syncthreads();
}

// k3: S[b,c,h,p,n] = sum_t x[t,p] * dt_t * exp(cs_end - cs_t) * B[t,g,n], plus
// the chunk's log-decay cs_end. grid (nchunks, H, batch).
template <typename T>
__global__ void __launch_bounds__(kThreads) simt_chunk_state(const T* __restrict__ x, const float* __restrict__ dt,
                                                             const float* __restrict__ dt_bias,
                                                             const float* __restrict__ A, const T* __restrict__ Bm,
                                                             int64_t L, int H, int G, int P, int N, int Q, int nc,
                                                             float* __restrict__ states,
                                                             float* __restrict__ chunk_logdecay, float2 lim,
                                                             const int32_t* __restrict__ seq) {
    extern __shared__ float sm[];
    float* s_dt = sm;
    float* s_cs = s_dt + kMaxChunk;
    float* s_warp = s_cs + kMaxChunk;
    float* s_w = s_warp + 8;                  // [Q] weights dt * exp(cs_end - cs)
    float* sx = s_w + kMaxChunk;              // [kRows][P]
    float* sb = sx + kRows * P;               // [kRows][N]

    const int c = blockIdx.x, h = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int g = h / (H / G);
    const int tid = threadIdx.x;
    chunk_dt_cumsum(dt, dt_bias, A, seq, b, h, c, Q, L, H, lim, s_dt, s_cs, s_warp);
    const float cs_end = s_cs[Q - 1];
    for (int t = tid; t < Q; t += kThreads) s_w[t] = s_dt[t] * expf(cs_end - s_cs[t]);
    if (tid == 0) chunk_logdecay[(b * H + h) * nc + c] = cs_end;
    __syncthreads();

    const int PN = P * N;
    float* out = states + ((b * nc + c) * H + h) * static_cast<int64_t>(PN);
    for (int base = 0; base < PN; base += kThreads * kAcc) {
        float acc[kAcc];
#pragma unroll
        for (int k = 0; k < kAcc; ++k) acc[k] = 0.f;
        for (int r0 = 0; r0 < Q; r0 += kRows) {
            __syncthreads();
            for (int i = tid; i < kRows * P; i += kThreads) {
                const int r = i / P, p = i % P;
                const int64_t t = static_cast<int64_t>(c) * Q + r0 + r;
                float v = 0.f;
                if (r0 + r < Q && t < L) v = load_f(x + ((b * L + t) * H + h) * P + p) * s_w[r0 + r];
                sx[i] = v;
            }
            for (int i = tid; i < kRows * N; i += kThreads) {
                const int r = i / N, n = i % N;
                const int64_t t = static_cast<int64_t>(c) * Q + r0 + r;
                sb[i] = (r0 + r < Q && t < L) ? load_f(Bm + ((b * L + t) * G + g) * N + n) : 0.f;
            }
            __syncthreads();
            const int rows = min(kRows, Q - r0);
#pragma unroll
            for (int k = 0; k < kAcc; ++k) {
                const int o = base + k * kThreads + tid;
                if (o < PN) {
                    const int p = o / N, n = o % N;
                    float a = acc[k];
                    for (int r = 0; r < rows; ++r) a = fmaf(sx[r * P + p], sb[r * N + n], a);
                    acc[k] = a;
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kAcc; ++k) {
            const int o = base + k * kThreads + tid;
            if (o < PN) out[o] = acc[k];
        }
    }
}

// k4: states[b,c,h] <- input state of chunk c; s_{c+1} = exp(cs_end_c) s_c + S_c.
// grid (ceil(P*N/256), H, batch).
__global__ void __launch_bounds__(kThreads) simt_state_pass(float* __restrict__ states,
                                                            const float* __restrict__ chunk_logdecay,
                                                            const float* __restrict__ init,
                                                            float* __restrict__ final_state, int H, int PN,
                                                            int nc) {
    const int h = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int e = blockIdx.x * kThreads + threadIdx.x;
    if (e >= PN) return;
    float s = init ? init[(b * H + h) * static_cast<int64_t>(PN) + e] : 0.f;
    for (int c = 0; c < nc; ++c) {
        float* slot = states + ((b * nc + c) * H + h) * static_cast<int64_t>(PN) + e;
        const float chunk_state = *slot;
        *slot = s;
        s = expf(chunk_logdecay[(b * H + h) * nc + c]) * s + chunk_state;
    }
    if (final_state) final_state[(b * H + h) * static_cast<int64_t>(PN) + e] = s;
}

// k2 + k5 for a 32-row tile of chunk c:
//   y[t,p] = exp(cs_t) C_t . s_in[p,:] + sum_{s<=t} (C_t . B_s) exp(cs_t - cs_s) dt_s x[s,p] + D x[t,p]
// grid (nchunks * ceil(Q/32), H, batch).
template <typename T>
__global__ void __launch_bounds__(kThreads) simt_chunk_scan(const T* __restrict__ x, const float* __restrict__ dt,
                                                            const float* __restrict__ dt_bias,
                                                            const float* __restrict__ A, const T* __restrict__ Bm,
                                                            const T* __restrict__ Cm, const float* __restrict__ D,
                                                            const float* __restrict__ states, int64_t L, int H,
                                                            int G, int P, int N, int Q, int nc, int tiles,
                                                            T* __restrict__ y, float2 lim,
                                                            const int32_t* __restrict__ seq) {
    extern __shared__ float sm[];
    float* s_dt = sm;
    float* s_cs = s_dt + kMaxChunk;
    float* s_warp = s_cs + kMaxChunk;
    float* sG = s_warp + 8;                   // [kRows][Q]
    float* sC = sG + kRows * kMaxChunk;       // [kRows][N]

    const int c = blockIdx.x / tiles, r0 = (blockIdx.x % tiles) * kRows;
    const int h = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int g = h / (H / G);
    const int tid = threadIdx.x;
    chunk_dt_cumsum(dt, dt_bias, A, seq, b, h, c, Q, L, H, lim, s_dt, s_cs, s_warp);

    const int rows = min(kRows, Q - r0);
    for (int i = tid; i < kRows * N; i += kThreads) {
        const int r = i / N, n = i % N;
        const int64_t t = static_cast<int64_t>(c) * Q + r0 + r;
        sC[i] = (r < rows && t < L) ? load_f(Cm + ((b * L + t) * G + g) * N + n) : 0.f;
    }
    __syncthreads();
    // masked, decayed C.B^T for the tile rows
    const int ncols = r0 + rows;  // causal: columns s <= last row of the tile
    for (int i = tid; i < rows * ncols; i += kThreads) {
        const int r = i / ncols, s = i % ncols;
        const int tl = r0 + r;
        float v = 0.f;
        if (s <= tl) {
            const int64_t ts = static_cast<int64_t>(c) * Q + s;
            if (ts < L) {
                const T* Bs = Bm + ((b * L + ts) * G + g) * N;
                const float* Cr = sC + r * N;
                float dot = 0.f;
                for (int n = 0; n < N; ++n) dot = fmaf(Cr[n], load_f(Bs + n), dot);
                v = dot * expf(s_cs[tl] - s_cs[s]) * s_dt[s];
            }
        }
        sG[r * kMaxChunk + s] = v;
    }
    __syncthreads();

    const float* s_in = states + ((b * nc + c) * H + h) * static_cast<int64_t>(P) * N;
    const float Dh = D ? D[h] : 0.f;
    for (int i = tid; i < rows * P; i += kThreads) {
        const int r = i / P, p = i % P;
        const int tl = r0 + r;
        const int64_t t = static_cast<int64_t>(c) * Q + tl;
        if (t >= L) continue;
        float off = 0.f;
        const float* sp = s_in + static_cast<int64_t>(p) * N;
        const float* Cr = sC + r * N;
        for (int n = 0; n < N; ++n) off = fmaf(Cr[n], sp[n], off);
        float diag = 0.f;
        for (int s = 0; s <= tl; ++s) {
            const int64_t ts = static_cast<int64_t>(c) * Q + s;
            diag = fmaf(sG[r * kMaxChunk + s], load_f(x + ((b * L + ts) * H + h) * P + p), diag);
        }
        const float xt = load_f(x + ((b * L + t) * H + h) * P + p);
        store_f(y + ((b * L + t) * H + h) * P + p, expf(s_cs[tl]) * off + diag + Dh * xt);
    }
}

template <typename T>
ssd_status launch_all(const FwdArgs& a, float* states, float* logdecay) {
    const ssd_dims& d = a.d;
    const int H = static_cast<int>(d.nheads), G = static_cast<int>(d.ngroups);
    const int P = static_cast<int>(d.headdim), N = static_cast<int>(d.dstate), Q = a.chunk_len;
    const int nc = static_cast<int>((d.seqlen + Q - 1) / Q);
    const dim3 block(kThreads);
    const T* x = static_cast<const T*>(a.x);
    const T* Bm = static_cast<const T*>(a.B);
    const T* Cm = static_cast<const T*>(a.C);

    const size_t smem1 = sizeof(float) * (3 * kMaxChunk + 8 + kRows * (P + N));
    const size_t smem3 = sizeof(float) * (2 * kMaxChunk + 8 + kRows * kMaxChunk + kRows * N);
    if (cudaFuncSetAttribute(simt_chunk_state<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem1)) != cudaSuccess ||
        cudaFuncSetAttribute(simt_chunk_scan<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem3)) != cudaSuccess)
        return SSD_ERR_CUDA;

    timing_begin(a.stream);
    simt_chunk_state<T><<<dim3(nc, H, static_cast<unsigned>(d.batch)), block, smem1, a.stream>>>(
        x, a.dt, a.dt_bias, a.A, Bm, d.seqlen, H, G, P, N, Q, nc, states, logdecay, make_float2(a.dt_min, a.dt_max),
        a.seq_idx);
    const int PN = P * N;
    simt_state_pass<<<dim3((PN + kThreads - 1) / kThreads, H, static_cast<unsigned>(d.batch)), block, 0,
                      a.stream>>>(states, logdecay, a.init, a.final_state, H, PN, nc);
    const int tiles = (Q + kRows - 1) / kRows;
    simt_chunk_scan<T><<<dim3(nc * tiles, H, static_cast<unsigned>(d.batch)), block, smem3, a.stream>>>(
        x, a.dt, a.dt_bias, a.A, Bm, Cm, a.D, states, d.seqlen, H, G, P, N, Q, nc, tiles,
        static_cast<T*>(a.y), make_float2(a.dt_min, a.dt_max), a.seq_idx);
    timing_end(a.stream);
    note_launches(3);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

bool simt_supported(const ssd_dims& d, int chunk_len) {
    return chunk_len >= 1 && chunk_len <= kMaxChunk && d.headdim <= 256 && d.dstate <= 256 &&
           d.nheads <= 65535 && d.batch <= 65535 && (d.seqlen + chunk_len - 1) / chunk_len * 8 <= (1ll << 31) - 1;
}

size_t simt_workspace_bytes(const ssd_dims& d, int chunk_len) {
    const int64_t nc = (d.seqlen + chunk_len - 1) / chunk_len;
    const size_t states = sizeof(float) * static_cast<size_t>(d.batch * nc * d.nheads * d.headdim * d.dstate);
    const size_t decay = sizeof(float) * static_cast<size_t>(d.batch * d.nheads * nc);
    return align_up(states, kWorkspaceAlign) + align_up(decay, kWorkspaceAlign);
}

ssd_status simt_forward(const FwdArgs& a, void* ws, size_t ws_bytes) {
    const int64_t nc = (a.d.seqlen + a.chunk_len - 1) / a.chunk_len;
    const size_t states_bytes =
        align_up(sizeof(float) * static_cast<size_t>(a.d.batch * nc * a.d.nheads * a.d.headdim * a.d.dstate),
                 kWorkspaceAlign);
    if (ws_bytes < simt_workspace_bytes(a.d, a.chunk_len)) return SSD_ERR_WORKSPACE;
    float* states = static_cast<float*>(ws);
    float* logdecay = reinterpret_cast<float*>(static_cast<char*>(ws) + states_bytes);
    if (a.io == SSD_F32) return launch_all<float>(a, states, logdecay);
    return launch_all<__nv_bfloat16>(a, states, logdecay);
}

}  // namespace ssd
