// One decode step of the SSM on a carried state (a single new token per
// sequence): fla "mamba2.py", Mamba2.torch_forward, cached-decode branch
// (the fast path calls selective_state_update):
//
//   dt' = clamp(softplus(dt + dt_bias[h]), dt_min, dt_max)   ((0, inf) by default)
//   state[p][n] = e^{dt' A[h]} state[p][n] + dt' x[p] B[n]     (in place, fp32)
//   y[p] = sum_n state[p][n] C[n] + D[h] x[p]
//
// The step reads and writes the whole fp32 state once: it is bound by HBM
// bandwidth, so the kernel is a plain streaming sweep. One CTA per (batch,
// head); each warp takes rows p, each lane four consecutive n (16-byte loads
// and stores, coalesced along n), and a warp reduction gives y[p]. For
// dstate 128 and 256 the lane's B and C stay in registers and four rows are
// loaded before any is written, to keep more loads in flight.
#include <cuda_bf16.h>

#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kStepThreads = 256;

__device__ __forceinline__ float load_io(const float* p, long long i) { return p[i]; }
__device__ __forceinline__ float load_io(const __nv_bfloat16* p, long long i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void store_io(float* p, long long i, float v) { p[i] = v; }
__device__ __forceinline__ void store_io(__nv_bfloat16* p, long long i, float v) { p[i] = __float2bfloat16_rn(v); }

__device__ __forceinline__ float softplus_step(float v) {
    return v > 0.f ? v + log1pf(expf(-v)) : log1pf(expf(v));
}

// n % 4 == 0: each lane owns groups of four consecutive state columns.
template <typename T>
__global__ void __launch_bounds__(kStepThreads)
    ssd_step_vec4(const T* __restrict__ x, const float* __restrict__ dt, const float* __restrict__ dt_bias,
                  const float* __restrict__ A, const T* __restrict__ B, const T* __restrict__ C,
                  const float* __restrict__ D, float* __restrict__ state, T* __restrict__ y, int H, int G, int P,
                  int N, float2 lim) {
    const int bh = blockIdx.x;
    const int b = bh / H, h = bh % H;
    const int g = h / (H / G);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float d = fminf(fmaxf(softplus_step(dt[bh] + dt_bias[h]), lim.x), lim.y);
    const float decay = expf(d * A[h]);
    const float Dh = D ? D[h] : 0.f;
    const long long bg = static_cast<long long>(b) * G + g;
    const int n4 = N / 4;
    float4* st = reinterpret_cast<float4*>(state + static_cast<long long>(bh) * P * N);
    for (int p = warp; p < P; p += kStepThreads / 32) {
        const float xp = load_io(x, static_cast<long long>(bh) * P + p);
        const float dx = d * xp;
        float acc = 0.f;
        for (int c4 = lane; c4 < n4; c4 += 32) {
            const long long nb = bg * N + 4 * c4;
            float4 s = st[p * n4 + c4];
            s.x = fmaf(decay, s.x, dx * load_io(B, nb + 0));
            s.y = fmaf(decay, s.y, dx * load_io(B, nb + 1));
            s.z = fmaf(decay, s.z, dx * load_io(B, nb + 2));
            s.w = fmaf(decay, s.w, dx * load_io(B, nb + 3));
            st[p * n4 + c4] = s;
            acc = fmaf(s.x, load_io(C, nb + 0), acc);
            acc = fmaf(s.y, load_io(C, nb + 1), acc);
            acc = fmaf(s.z, load_io(C, nb + 2), acc);
            acc = fmaf(s.w, load_io(C, nb + 3), acc);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) store_io(y, static_cast<long long>(bh) * P + p, fmaf(Dh, xp, acc));
    }
}

// n = 128 * NV: lane l owns column groups l, l + 32, ... (four columns each);
// B and C for them stay in registers, and four rows are in flight per warp.
template <typename T, int NV>
__global__ void __launch_bounds__(kStepThreads)
    ssd_step_rows4(const T* __restrict__ x, const float* __restrict__ dt, const float* __restrict__ dt_bias,
                   const float* __restrict__ A, const T* __restrict__ B, const T* __restrict__ C,
                   const float* __restrict__ D, float* __restrict__ state, T* __restrict__ y, int H, int G, int P, float2 lim) {
    constexpr int N = 128 * NV, N4 = N / 4;
    const int bh = blockIdx.x;
    const int b = bh / H, h = bh % H;
    const int g = h / (H / G);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float d = fminf(fmaxf(softplus_step(dt[bh] + dt_bias[h]), lim.x), lim.y);
    const float decay = expf(d * A[h]);
    const float Dh = D ? D[h] : 0.f;
    const long long bg = static_cast<long long>(b) * G + g;
    float4 bv[NV], cv[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const long long nb = bg * N + 4 * (lane + 32 * v);
        bv[v] = make_float4(load_io(B, nb), load_io(B, nb + 1), load_io(B, nb + 2), load_io(B, nb + 3));
        cv[v] = make_float4(load_io(C, nb), load_io(C, nb + 1), load_io(C, nb + 2), load_io(C, nb + 3));
    }
    float4* st = reinterpret_cast<float4*>(state + static_cast<long long>(bh) * P * N);
    constexpr int RW = 4;  // rows per warp step
    for (int p0 = warp * RW; p0 < P; p0 += (kStepThreads / 32) * RW) {
        float4 sv[RW][NV];
        float xr[RW];
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            const int p = p0 + r;
            xr[r] = p < P ? load_io(x, static_cast<long long>(bh) * P + p) : 0.f;
#pragma unroll
            for (int v = 0; v < NV; ++v) sv[r][v] = p < P ? st[p * N4 + lane + 32 * v] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float acc[RW];
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            const float dx = d * xr[r];
            acc[r] = 0.f;
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                float4 s4 = sv[r][v];
                s4.x = fmaf(decay, s4.x, dx * bv[v].x);
                s4.y = fmaf(decay, s4.y, dx * bv[v].y);
                s4.z = fmaf(decay, s4.z, dx * bv[v].z);
                s4.w = fmaf(decay, s4.w, dx * bv[v].w);
                if (p0 + r < P) st[(p0 + r) * N4 + lane + 32 * v] = s4;
                acc[r] = fmaf(s4.x, cv[v].x, fmaf(s4.y, cv[v].y, fmaf(s4.z, cv[v].z, fmaf(s4.w, cv[v].w, acc[r]))));
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int r = 0; r < RW; ++r) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
        if (lane < RW && p0 + lane < P) {
            float a = acc[0], xp = xr[0];
#pragma unroll
            for (int r = 1; r < RW; ++r) {
                a = lane == r ? acc[r] : a;
                xp = lane == r ? xr[r] : xp;
            }
            store_io(y, static_cast<long long>(bh) * P + p0 + lane, fmaf(Dh, xp, a));
        }
    }
}

// Any n: one state element per lane step.
template <typename T>
__global__ void __launch_bounds__(kStepThreads)
    ssd_step_scalar(const T* __restrict__ x, const float* __restrict__ dt, const float* __restrict__ dt_bias,
                    const float* __restrict__ A, const T* __restrict__ B, const T* __restrict__ C,
                    const float* __restrict__ D, float* __restrict__ state, T* __restrict__ y, int H, int G, int P,
                    int N, float2 lim) {
    const int bh = blockIdx.x;
    const int b = bh / H, h = bh % H;
    const int g = h / (H / G);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float d = fminf(fmaxf(softplus_step(dt[bh] + dt_bias[h]), lim.x), lim.y);
    const float decay = expf(d * A[h]);
    const float Dh = D ? D[h] : 0.f;
    const long long bg = static_cast<long long>(b) * G + g;
    float* st = state + static_cast<long long>(bh) * P * N;
    for (int p = warp; p < P; p += kStepThreads / 32) {
        const float xp = load_io(x, static_cast<long long>(bh) * P + p);
        const float dx = d * xp;
        float acc = 0.f;
        for (int n = lane; n < N; n += 32) {
            const float s = fmaf(decay, st[static_cast<long long>(p) * N + n], dx * load_io(B, bg * N + n));
            st[static_cast<long long>(p) * N + n] = s;
            acc = fmaf(s, load_io(C, bg * N + n), acc);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) store_io(y, static_cast<long long>(bh) * P + p, fmaf(Dh, xp, acc));
    }
}

template <typename T>
ssd_status launch_step(const StepArgs& a) {
    const ssd_dims& d = a.d;
    const unsigned grid = static_cast<unsigned>(d.batch * d.nheads);
    const int H = static_cast<int>(d.nheads), G = static_cast<int>(d.ngroups), P = static_cast<int>(d.headdim),
              N = static_cast<int>(d.dstate);
    const T* x = static_cast<const T*>(a.x);
    const T* B = static_cast<const T*>(a.B);
    const T* C = static_cast<const T*>(a.C);
    T* y = static_cast<T*>(a.y);
    const float2 lim = make_float2(a.dt_min, a.dt_max);
    if (N == 128)
        ssd_step_rows4<T, 1><<<grid, kStepThreads, 0, a.stream>>>(x, a.dt, a.dt_bias, a.A, B, C, a.D, a.state, y, H, G, P, lim);
    else if (N == 256)
        ssd_step_rows4<T, 2><<<grid, kStepThreads, 0, a.stream>>>(x, a.dt, a.dt_bias, a.A, B, C, a.D, a.state, y, H, G, P, lim);
    else if (N % 4 == 0)
        ssd_step_vec4<T><<<grid, kStepThreads, 0, a.stream>>>(x, a.dt, a.dt_bias, a.A, B, C, a.D, a.state, y, H, G, P, N, lim);
    else
        ssd_step_scalar<T><<<grid, kStepThreads, 0, a.stream>>>(x, a.dt, a.dt_bias, a.A, B, C, a.D, a.state, y, H, G,
                                                                P, N, lim);
    note_launches(1);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

bool step_supported(const ssd_dims& d) {
    return d.batch * d.nheads < (1ll << 31) && d.headdim < (1 << 20) && d.dstate < (1 << 20) &&
           d.batch * d.nheads * d.headdim * d.dstate < (1ll << 40);
}

ssd_status step_forward(const StepArgs& a) {
    if (a.io == SSD_BF16) return launch_step<__nv_bfloat16>(a);
    return launch_step<float>(a);
}

}  // namespace ssd
