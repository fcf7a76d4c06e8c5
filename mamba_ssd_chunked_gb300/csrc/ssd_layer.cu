// The per-token operations around the SSD scan in a Mamba-2 layer (fla
// "mamba2.py", Mamba2.torch_forward steps 2 and 3):
//
//   ssd_conv1d_silu   causal depthwise conv1d over time + SiLU of the in_proj
//                     slice xBC, split into x, B and C (the scan's inputs);
//                     optionally the last kernel_size inputs as conv state
//   ssd_conv1d_step   the cached-decode form: shift the conv state, append the
//                     new token, one output per channel
//   ssd_gated_rmsnorm RMSNormGated with norm_before_gate=False applied to the
//                     scan output and the gate z
//
// All three read and write each element once and do a few flops per element:
// they are bound by HBM bandwidth. The kernels are plain streaming sweeps with
// 16-byte accesses along the channel dimension (coalesced across a warp) and
// fp32 arithmetic; rows may be strided so xBC and z can be read straight out of
// the in_proj output.
#include <cuda_bf16.h>

#include "ssd_internal.h"

namespace ssd {
namespace {

// ---------------------------------------------------------------- element I/O
template <typename T>
struct Io;
template <>
struct Io<float> {
    static constexpr int kVec = 4;  // elements per 16 bytes
    __device__ static float ld(const float* p) { return *p; }
    __device__ static void st(float* p, float v) { *p = v; }
    __device__ static void ldv(const float* p, float* f) {
        const float4 v = *reinterpret_cast<const float4*>(p);
        f[0] = v.x, f[1] = v.y, f[2] = v.z, f[3] = v.w;
    }
    __device__ static void stv(float* p, const float* f) {
        *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
    }
};
template <>
struct Io<__nv_bfloat16> {
    static constexpr int kVec = 8;
    __device__ static float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
    __device__ static void st(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
    __device__ static void ldv(const __nv_bfloat16* p, float* f) {
        const uint4 v = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    __device__ static void stv(__nv_bfloat16* p, const float* f) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// V elements starting at p: one 16-byte access when V is the vector width, else scalars.
template <typename T, int V>
__device__ __forceinline__ void load_n(const T* p, float* f) {
    if constexpr (V == Io<T>::kVec) {
        Io<T>::ldv(p, f);
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i) f[i] = Io<T>::ld(p + i);
    }
}
template <typename T, int V>
__device__ __forceinline__ void store_n(T* p, const float* f) {
    if constexpr (V == Io<T>::kVec) {
        Io<T>::stv(p, f);
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i) Io<T>::st(p + i, f[i]);
    }
}

__device__ __forceinline__ float silu_f(float v) { return __fdividef(v, 1.f + __expf(-v)); }

// SiLU with one MUFU op: v * sigmoid(v) = h + h * tanh(h), h = v / 2. tanh.approx
// has a relative error near 2^-11, far below bf16 rounding; fp32 outputs use silu_f.
__device__ __forceinline__ float silu_tanh(float v) {
    const float h = 0.5f * v;
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
    return fmaf(h, t, h);
}

template <typename T>
__device__ __forceinline__ float silu_io(float v) {
    if constexpr (sizeof(T) == 2) {
        return silu_tanh(v);
    } else {
        return silu_f(v);
    }
}

// V raw elements of T, moved with one access of V * sizeof(T) bytes when that
// is 4, 8 or 16 (the pointer is then aligned to it), else element by element.
template <typename T, int V>
struct Raw {
    static constexpr int kBytes = V * static_cast<int>(sizeof(T));
    static constexpr int kWords = kBytes >= 4 ? kBytes / 4 : 1;
    uint32_t w[kWords];
    __device__ __forceinline__ void load(const T* p) {
        if constexpr (kBytes == 16) {
            const uint4 v = *reinterpret_cast<const uint4*>(p);
            w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
        } else if constexpr (kBytes == 8) {
            const uint2 v = *reinterpret_cast<const uint2*>(p);
            w[0] = v.x, w[1] = v.y;
        } else if constexpr (kBytes == 4) {
            w[0] = *reinterpret_cast<const uint32_t*>(p);
        } else {
            w[0] = *reinterpret_cast<const uint16_t*>(p);
        }
    }
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int i = 0; i < kWords; ++i) w[i] = 0u;
    }
    __device__ __forceinline__ float get(int i) const {
        if constexpr (sizeof(T) == 2) {
            const uint32_t u = w[i >> 1];
            return __uint_as_float((i & 1) ? (u & 0xFFFF0000u) : (u << 16));
        } else {
            return __uint_as_float(w[i]);
        }
    }
};

template <typename T, int V>
__device__ __forceinline__ void store_raw(T* p, const float* f) {
    constexpr int kBytes = V * static_cast<int>(sizeof(T));
    if constexpr (sizeof(T) == 2 && (kBytes == 16 || kBytes == 8 || kBytes == 4)) {
        uint32_t w[kBytes / 4];
#pragma unroll
        for (int i = 0; i < kBytes / 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        if constexpr (kBytes == 16)
            *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
        else if constexpr (kBytes == 8)
            *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
        else
            *reinterpret_cast<uint32_t*>(p) = w[0];
    } else if constexpr (sizeof(T) == 4 && kBytes == 16) {
        *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
    } else if constexpr (sizeof(T) == 4 && kBytes == 8) {
        *reinterpret_cast<float2*>(p) = make_float2(f[0], f[1]);
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i) Io<T>::st(p + i, f[i]);
    }
}

struct ConvShape {
    long long L, stride;  // tokens, elements between consecutive tokens of xBC
    int cd, d_inner, gn;  // channels: conv_dim = d_inner + 2 gn
    int act;              // 1: SiLU
};

// Output channel c goes to x, B or C (c is V-aligned and the three ranges are
// multiples of V, so a vector never straddles two of them): base and row length.
template <typename T>
__device__ __forceinline__ T* out_base(T* x, T* B, T* C, const ConvShape& s, int c, int* row) {
    if (c < s.d_inner) {
        *row = s.d_inner;
        return x + c;
    }
    c -= s.d_inner;
    *row = s.gn;
    return c < s.gn ? B + c : C + (c - s.gn);
}

constexpr int kConvThreads = 128;
constexpr int kConvRun = 32;  // tokens per thread
constexpr int kConvGroup = 8; // tokens loaded together; the next group is in flight during compute

// One thread: V consecutive channels of one batch row over kConvRun tokens. The
// previous K - 1 inputs stay in registers (raw io values) as a sliding window,
// and the loads of the next kConvGroup tokens are issued before the current
// group is computed.
template <typename T, int V, int K>
__global__ void __launch_bounds__(kConvThreads)
    conv1d_fwd(const T* __restrict__ xbc, const float* __restrict__ w, const float* __restrict__ bias,
               T* __restrict__ x, T* __restrict__ B, T* __restrict__ C, T* __restrict__ state, ConvShape s) {
    const int c = (blockIdx.x * kConvThreads + threadIdx.x) * V;
    if (c >= s.cd) return;
    const long long b = blockIdx.z;
    const int t0 = static_cast<int>(blockIdx.y) * kConvRun;
    const int t1 = static_cast<int>(t0 + kConvRun < s.L ? t0 + kConvRun : s.L);
    const T* in = xbc + b * s.L * s.stride + c;
    int orow;
    T* out = out_base(x, B, C, s, c, &orow) + b * s.L * orow;
    float wk[K][V], bv[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
#pragma unroll
        for (int k = 0; k < K; ++k) wk[k][i] = w[(c + i) * K + k];
        bv[i] = bias ? bias[c + i] : 0.f;
    }
    Raw<T, V> win[K];  // win[k]: input at token t - (K - 1) + k while token t is computed
#pragma unroll
    for (int k = 0; k < K - 1; ++k) {
        const int t = t0 - (K - 1) + k;
        if (t >= 0)
            win[k].load(in + static_cast<long long>(t) * s.stride);
        else
            win[k].zero();
    }
    Raw<T, V> cur[kConvGroup], nxt[kConvGroup];
#pragma unroll
    for (int a = 0; a < kConvGroup; ++a)
        if (t0 + a < t1) cur[a].load(in + static_cast<long long>(t0 + a) * s.stride);
    for (int tb = t0; tb < t1; tb += kConvGroup) {
#pragma unroll
        for (int a = 0; a < kConvGroup; ++a)
            if (tb + kConvGroup + a < t1) nxt[a].load(in + static_cast<long long>(tb + kConvGroup + a) * s.stride);
#pragma unroll
        for (int a = 0; a < kConvGroup; ++a) {
            if (tb + a < t1) {
                win[K - 1] = cur[a];
                float o[V];
#pragma unroll
                for (int i = 0; i < V; ++i) {
                    float acc = bv[i];
#pragma unroll
                    for (int k = 0; k < K; ++k) acc = fmaf(wk[k][i], win[k].get(i), acc);
                    o[i] = s.act ? silu_io<T>(acc) : acc;
                }
                store_raw<T, V>(out + static_cast<long long>(tb + a) * orow, o);
#pragma unroll
                for (int k = 0; k < K - 1; ++k) win[k] = win[k + 1];
            }
        }
#pragma unroll
        for (int a = 0; a < kConvGroup; ++a) cur[a] = nxt[a];
    }
    // conv state: the last K inputs, channel-major [b][cd][K], zeros before the sequence
    if (state && t1 == s.L) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const long long t = s.L - K + k;
            Raw<T, V> v;
            if (t >= 0)
                v.load(in + t * s.stride);
            else
                v.zero();
#pragma unroll
            for (int i = 0; i < V; ++i) Io<T>::st(state + (b * s.cd + c + i) * K + k, v.get(i));
        }
    }
}

// One thread: V channels of one sequence; state [b][cd][K] shifted in place.
template <typename T, int V, int K>
__global__ void __launch_bounds__(kConvThreads)
    conv1d_step(const T* __restrict__ xbc, const float* __restrict__ w, const float* __restrict__ bias,
                T* __restrict__ x, T* __restrict__ B, T* __restrict__ C, T* __restrict__ state, ConvShape s) {
    const int c = (blockIdx.x * kConvThreads + threadIdx.x) * V;
    if (c >= s.cd) return;
    const long long b = blockIdx.y;
    Raw<T, V> cur;
    cur.load(xbc + b * s.stride + c);
    float o[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
        T* st = state + (b * s.cd + c + i) * K;
        float acc = bias ? bias[c + i] : 0.f;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const float v = k + 1 < K ? Io<T>::ld(st + k + 1) : cur.get(i);
            acc = fmaf(w[(c + i) * K + k], v, acc);
            Io<T>::st(st + k, v);
        }
        o[i] = s.act ? silu_io<T>(acc) : acc;
    }
    int orow;
    T* out = out_base(x, B, C, s, c, &orow) + b * orow;
    store_raw<T, V>(out, o);
}

template <typename T, int V>
ssd_status launch_conv(bool step, int K, const void* xbc, const float* w, const float* bias, void* x, void* B,
                       void* C, void* state, const ConvShape& s, long long batch, cudaStream_t stream) {
    const unsigned gx = static_cast<unsigned>((s.cd / V + kConvThreads - 1) / kConvThreads);
    const dim3 grid = step ? dim3(gx, static_cast<unsigned>(batch), 1)
                           : dim3(gx, static_cast<unsigned>((s.L + kConvRun - 1) / kConvRun),
                                  static_cast<unsigned>(batch));
    const T* in = static_cast<const T*>(xbc);
    T *xo = static_cast<T*>(x), *bo = static_cast<T*>(B), *co = static_cast<T*>(C), *so = static_cast<T*>(state);
#define SSD_CONV_CASE(KK)                                                                                 \
    case KK:                                                                                              \
        if (step)                                                                                         \
            conv1d_step<T, V, KK><<<grid, kConvThreads, 0, stream>>>(in, w, bias, xo, bo, co, so, s);     \
        else                                                                                              \
            conv1d_fwd<T, V, KK><<<grid, kConvThreads, 0, stream>>>(in, w, bias, xo, bo, co, so, s);      \
        break;
    switch (K) {
        SSD_CONV_CASE(1)
        SSD_CONV_CASE(2)
        SSD_CONV_CASE(3)
        SSD_CONV_CASE(4)
        SSD_CONV_CASE(5)
        SSD_CONV_CASE(6)
        SSD_CONV_CASE(7)
        SSD_CONV_CASE(8)
        default:
            return SSD_ERR_UNSUPPORTED;
    }
#undef SSD_CONV_CASE
    note_launches(1);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

// ---------------------------------------------------------------- gated RMSNorm
constexpr int kNormThreads = 128;
constexpr int kNormMaxGroups = 64;

struct NormShape {
    long long dim, group, ystride, zstride, ostride;
    float eps;
};

// One CTA per row. R > 0: the row's gated values stay in registers (R vectors
// per thread); R == 0: the second pass reads y and z again (L1/L2 hits).
template <typename T, int V, int R>
__global__ void __launch_bounds__(kNormThreads)
    gated_rmsnorm(const T* __restrict__ y, const T* __restrict__ z, const float* __restrict__ w,
                  T* __restrict__ out, NormShape s) {
    __shared__ float sums[kNormMaxGroups];
    __shared__ float warp_sums[kNormThreads / 32];
    const long long row = blockIdx.x;
    const T* yr = y + row * s.ystride;
    const T* zr = z ? z + row * s.zstride : nullptr;
    T* orow = out + row * s.ostride;
    const int ngroups = static_cast<int>(s.dim / s.group);
    const int group = static_cast<int>(s.group);  // dim < 2^30: 32-bit channel indices
    const int nvec = static_cast<int>(s.dim / V);
    for (int g = threadIdx.x; g < ngroups; g += kNormThreads) sums[g] = 0.f;
    __syncthreads();

    auto gated = [&](int vi, float* v) {
        load_n<T, V>(yr + static_cast<long long>(vi) * V, v);
        if (zr) {
            float g[V];
            load_n<T, V>(zr + static_cast<long long>(vi) * V, g);
#pragma unroll
            for (int i = 0; i < V; ++i) v[i] *= silu_io<T>(g[i]);
        }
    };
    // pass 1: gated values and their squares summed per group
    float keep[R > 0 ? R : 1][V];
    float tot = 0.f;  // one group: this thread's partial sum
    auto accumulate = [&](int vi, const float* v) {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < V; ++i) ss = fmaf(v[i], v[i], ss);
        if (ngroups == 1)
            tot += ss;
        else
            atomicAdd(&sums[vi * V / group], ss);
    };
    if constexpr (R > 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int vi = threadIdx.x + r * kNormThreads;
            if (vi < nvec) {
                gated(vi, keep[r]);
                accumulate(vi, keep[r]);
            }
        }
    } else {
        for (int vi = threadIdx.x; vi < nvec; vi += kNormThreads) {
            float v[V];
            gated(vi, v);
            accumulate(vi, v);
        }
    }
    if (ngroups == 1) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
        if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = tot;
    }
    __syncthreads();
    if (ngroups == 1 && threadIdx.x == 0) {
        float a = 0.f;
#pragma unroll
        for (int i = 0; i < kNormThreads / 32; ++i) a += warp_sums[i];
        sums[0] = a;
    }
    __syncthreads();
    // pass 2: scale by the group's 1/rms and the weight
    const float inv_group = 1.f / static_cast<float>(s.group);
    const float rstd0 = rsqrtf(fmaf(sums[0], inv_group, s.eps));
    auto emit = [&](int vi, const float* v) {
        const float rstd = ngroups == 1 ? rstd0 : rsqrtf(fmaf(sums[vi * V / group], inv_group, s.eps));
        float wv[V];
        if constexpr (V % 4 == 0) {
            const float4* w4 = reinterpret_cast<const float4*>(w + static_cast<long long>(vi) * V);
#pragma unroll
            for (int i = 0; i < V / 4; ++i) {
                const float4 q = w4[i];
                wv[4 * i] = q.x, wv[4 * i + 1] = q.y, wv[4 * i + 2] = q.z, wv[4 * i + 3] = q.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < V; ++i) wv[i] = w[static_cast<long long>(vi) * V + i];
        }
        float o[V];
#pragma unroll
        for (int i = 0; i < V; ++i) o[i] = v[i] * rstd * wv[i];
        store_n<T, V>(orow + static_cast<long long>(vi) * V, o);
    };
    if constexpr (R > 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int vi = threadIdx.x + r * kNormThreads;
            if (vi < nvec) emit(vi, keep[r]);
        }
    } else {
        for (int vi = threadIdx.x; vi < nvec; vi += kNormThreads) {
            float v[V];
            gated(vi, v);
            emit(vi, v);
        }
    }
}

template <typename T, int V>
ssd_status launch_norm(long long rows, const void* y, const void* z, const float* w, void* out, const NormShape& s,
                       cudaStream_t stream) {
    const long long per_thread = (s.dim / V + kNormThreads - 1) / kNormThreads;
    const T* yi = static_cast<const T*>(y);
    const T* zi = static_cast<const T*>(z);
    T* o = static_cast<T*>(out);
    const unsigned grid = static_cast<unsigned>(rows);
    switch (per_thread) {
#define SSD_NORM_CASE(RR) \
    case RR:              \
        gated_rmsnorm<T, V, RR><<<grid, kNormThreads, 0, stream>>>(yi, zi, w, o, s); \
        break;
        SSD_NORM_CASE(1)
        SSD_NORM_CASE(2)
        SSD_NORM_CASE(3)
        SSD_NORM_CASE(4)
        SSD_NORM_CASE(5)
        SSD_NORM_CASE(6)
        SSD_NORM_CASE(7)
        SSD_NORM_CASE(8)
#undef SSD_NORM_CASE
        default:
            gated_rmsnorm<T, V, 0><<<grid, kNormThreads, 0, stream>>>(yi, zi, w, o, s);
    }
    note_launches(1);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

ssd_status check_conv(const ssd_conv_dims* d, ssd_dtype io, const void* xbc, int64_t stride, const float* w,
                      const void* x, const void* B, const void* C) {
    if (!d || !xbc || !w || !x || !B || !C) return SSD_ERR_INVALID_ARG;
    if (io != SSD_F32 && io != SSD_BF16) return SSD_ERR_INVALID_ARG;
    if (d->batch < 1 || d->seqlen < 1 || d->d_inner < 1 || d->ngroups < 1 || d->dstate < 1 || d->kernel_size < 1)
        return SSD_ERR_INVALID_ARG;
    const int64_t cd = d->d_inner + 2 * d->ngroups * d->dstate;
    if (stride < cd) return SSD_ERR_INVALID_ARG;
    if (d->kernel_size > 8) return SSD_ERR_UNSUPPORTED;
    if (cd >= (1ll << 30) || d->batch >= 65536 || d->batch * d->seqlen * stride >= (1ll << 60))
        return SSD_ERR_UNSUPPORTED;
    const size_t es = io == SSD_BF16 ? 2 : 4;
    for (const void* p : {xbc, static_cast<const void*>(w), static_cast<const void*>(x), static_cast<const void*>(B),
                          static_cast<const void*>(C)})
        if (!aligned(p, es < 4 ? 4 : es)) return SSD_ERR_UNSUPPORTED;
    return SSD_OK;
}

// The vector path moves 4 channels per access (8 bytes bf16, 16 bytes fp32): every
// row start and every x/B/C boundary must sit on that access size. Four bf16
// channels per thread measured faster than eight (fewer registers per thread,
// more warps per SM).
bool conv_vec_ok(const ssd_conv_dims* d, ssd_dtype io, const void* xbc, int64_t stride, const void* x,
                 const void* B, const void* C) {
    const size_t bytes = io == SSD_BF16 ? 8 : 16;
    const int64_t gn = d->ngroups * d->dstate;
    return d->d_inner % 4 == 0 && gn % 4 == 0 && stride % 4 == 0 && aligned(xbc, bytes) && aligned(x, bytes) &&
           aligned(B, bytes) && aligned(C, bytes);
}

ssd_status run_conv(bool step, const ssd_conv_dims* d, ssd_dtype io, const void* xbc, int64_t stride,
                    const float* w, const float* bias, int activation, void* x, void* B, void* C, void* state,
                    void* stream) {
    ConvShape s;
    s.L = step ? 1 : d->seqlen;
    s.stride = stride;
    s.d_inner = static_cast<int>(d->d_inner);
    s.gn = static_cast<int>(d->ngroups * d->dstate);
    s.cd = s.d_inner + 2 * s.gn;
    s.act = activation ? 1 : 0;
    const bool vec = conv_vec_ok(d, io, xbc, stride, x, B, C);
    const int K = static_cast<int>(d->kernel_size);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (io == SSD_BF16)
        return vec ? launch_conv<__nv_bfloat16, 4>(step, K, xbc, w, bias, x, B, C, state, s, d->batch, st)
                   : launch_conv<__nv_bfloat16, 1>(step, K, xbc, w, bias, x, B, C, state, s, d->batch, st);
    return vec ? launch_conv<float, 4>(step, K, xbc, w, bias, x, B, C, state, s, d->batch, st)
               : launch_conv<float, 1>(step, K, xbc, w, bias, x, B, C, state, s, d->batch, st);
}

}  // namespace
}  // namespace ssd

extern "C" {

ssd_status ssd_conv1d_silu(const ssd_conv_dims* dims, ssd_dtype io_dtype, const void* xbc, int64_t xbc_row_stride,
                           const float* weight, const float* bias, int activation, void* x, void* B, void* C,
                           void* conv_state, void* stream) {
    using namespace ssd;
    ssd_status st = check_conv(dims, io_dtype, xbc, xbc_row_stride, weight, x, B, C);
    if (st != SSD_OK) return st;
    if (dims->seqlen >= (1ll << 31) / 2) return SSD_ERR_UNSUPPORTED;
    const size_t es = io_dtype == SSD_BF16 ? 2 : 4;
    if (conv_state && !aligned(conv_state, es)) return SSD_ERR_UNSUPPORTED;
    if (bias && !aligned(bias, 4)) return SSD_ERR_UNSUPPORTED;
    return run_conv(false, dims, io_dtype, xbc, xbc_row_stride, weight, bias, activation, x, B, C, conv_state,
                    stream);
}

ssd_status ssd_conv1d_step(const ssd_conv_dims* dims, ssd_dtype io_dtype, const void* xbc, int64_t xbc_row_stride,
                           const float* weight, const float* bias, int activation, void* conv_state, void* x,
                           void* B, void* C, void* stream) {
    using namespace ssd;
    ssd_status st = check_conv(dims, io_dtype, xbc, xbc_row_stride, weight, x, B, C);
    if (st != SSD_OK) return st;
    if (dims->seqlen != 1 || !conv_state) return SSD_ERR_INVALID_ARG;
    const size_t es = io_dtype == SSD_BF16 ? 2 : 4;
    if (!aligned(conv_state, es)) return SSD_ERR_UNSUPPORTED;
    if (bias && !aligned(bias, 4)) return SSD_ERR_UNSUPPORTED;
    return run_conv(true, dims, io_dtype, xbc, xbc_row_stride, weight, bias, activation, x, B, C, conv_state,
                    stream);
}

ssd_status ssd_gated_rmsnorm(ssd_dtype io_dtype, int64_t rows, int64_t dim, int64_t group_size, const void* y,
                             int64_t y_row_stride, const void* z, int64_t z_row_stride, const float* weight,
                             float eps, void* out, int64_t out_row_stride, void* stream) {
    using namespace ssd;
    if (io_dtype != SSD_F32 && io_dtype != SSD_BF16) return SSD_ERR_INVALID_ARG;
    if (!y || !weight || !out || rows < 1 || dim < 1) return SSD_ERR_INVALID_ARG;
    const int64_t gs = group_size > 0 ? group_size : dim;
    if (dim % gs != 0) return SSD_ERR_INVALID_ARG;
    if (y_row_stride < dim || out_row_stride < dim || (z && z_row_stride < dim)) return SSD_ERR_INVALID_ARG;
    if (!(eps >= 0.f)) return SSD_ERR_INVALID_ARG;
    if (dim / gs > kNormMaxGroups || rows >= (1ll << 31) || dim >= (1ll << 30)) return SSD_ERR_UNSUPPORTED;
    const size_t es = io_dtype == SSD_BF16 ? 2 : 4;
    for (const void* p : {y, static_cast<const void*>(weight), static_cast<const void*>(out), z})
        if (p && !aligned(p, es < 4 ? 4 : es)) return SSD_ERR_UNSUPPORTED;
    const int64_t v = io_dtype == SSD_BF16 ? 8 : 4;
    const bool vec = dim % v == 0 && gs % v == 0 && y_row_stride % v == 0 && out_row_stride % v == 0 &&
                     (!z || z_row_stride % v == 0) && aligned(y, 16) && aligned(out, 16) && (!z || aligned(z, 16)) &&
                     aligned(weight, 16);
    NormShape s;
    s.dim = dim;
    s.group = gs;
    s.ystride = y_row_stride;
    s.zstride = z ? z_row_stride : 0;
    s.ostride = out_row_stride;
    s.eps = eps;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (io_dtype == SSD_BF16)
        return vec ? launch_norm<__nv_bfloat16, 8>(rows, y, z, weight, out, s, st)
                   : launch_norm<__nv_bfloat16, 1>(rows, y, z, weight, out, s, st);
    return vec ? launch_norm<float, 4>(rows, y, z, weight, out, s, st)
               : launch_norm<float, 1>(rows, y, z, weight, out, s, st);
}

}  // extern "C"
