// The input guard (ssd_check_inputs): counts the non-finite elements of each
// input of a forward. The burn-mamba port checks every input tensor before its
// kernels run (`mamba2/ssd/serial.rs`, Mamba2::ssd_serial, the sanity calls on
// x, dt, A, B, C, D and the initial state); a NaN or an infinity in any of them
// spreads through the state to every later token of its chain.
//
// One launch covers all eight tensors: blockIdx.y picks the tensor, the blocks
// along x stride over it with 16-byte loads (scalar loads for the unaligned head
// and the tail). An element is non-finite when its exponent bits are all ones
// (IEEE binary32 and bfloat16 alike: NaN and both infinities), a test on the
// bits alone. HBM bound: one read of every input.
#include <algorithm>

#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kGuardThreads = 256;
constexpr int kGuardTensors = 8;

struct GuardSpan {
    const void* p;  // null: absent optional input, counted as 0
    long long n;    // elements
    int bf16;       // element type: bfloat16 (else fp32)
};

struct GuardArgs {
    GuardSpan s[kGuardTensors];
    unsigned long long* counts;  // device [kGuardTensors], zeroed before the launch
};

__device__ __forceinline__ unsigned bad_f32(uint32_t w) { return (w & 0x7f800000u) == 0x7f800000u ? 1u : 0u; }
__device__ __forceinline__ unsigned bad_bf16x2(uint32_t w) {
    return ((w & 0x7f80u) == 0x7f80u ? 1u : 0u) + ((w & 0x7f800000u) == 0x7f800000u ? 1u : 0u);
}
__device__ __forceinline__ unsigned bad_bf16(uint16_t v) { return (v & 0x7f80u) == 0x7f80u ? 1u : 0u; }

__global__ void __launch_bounds__(kGuardThreads) count_nonfinite(const GuardArgs a) {
    const GuardSpan sp = a.s[blockIdx.y];
    if (sp.p == nullptr || sp.n <= 0) return;
    const int esz = sp.bf16 ? 2 : 4;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(sp.p);
    // elements before the first 16-byte boundary (the pointer is element-aligned)
    const long long head = min(sp.n, static_cast<long long>(((16u - (addr & 15u)) & 15u) / esz));
    const long long per = 16 / esz;
    const long long nvec = (sp.n - head) / per;
    const long long tail0 = head + nvec * per;
    const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long nthr = static_cast<long long>(gridDim.x) * blockDim.x;
    unsigned c = 0;
    auto scalar = [&](long long i) {
        if (sp.bf16)
            c += bad_bf16(__ldg(static_cast<const uint16_t*>(sp.p) + i));
        else
            c += bad_f32(__ldg(static_cast<const uint32_t*>(sp.p) + i));
    };
    if (tid < head) scalar(tid);
    const uint4* v = reinterpret_cast<const uint4*>(static_cast<const char*>(sp.p) + head * esz);
    // a thread's count stays far below 2^32: at most 8 per 16-byte load
    for (long long i = tid; i < nvec; i += nthr) {
        const uint4 w = __ldg(v + i);
        c += sp.bf16 ? bad_bf16x2(w.x) + bad_bf16x2(w.y) + bad_bf16x2(w.z) + bad_bf16x2(w.w)
                     : bad_f32(w.x) + bad_f32(w.y) + bad_f32(w.z) + bad_f32(w.w);
    }
    if (tid < sp.n - tail0) scalar(tail0 + tid);
    c = __reduce_add_sync(0xffffffffu, c);
    if ((threadIdx.x & 31) == 0 && c != 0) atomicAdd(a.counts + blockIdx.y, static_cast<unsigned long long>(c));
}

}  // namespace

ssd_status check_inputs(const CheckArgs& a, int64_t* counts) {
    GuardArgs g;
    const long long b = a.d.batch, L = a.d.seqlen, h = a.d.nheads, p = a.d.headdim, gr = a.d.ngroups,
                    n = a.d.dstate;
    const int io16 = a.io == SSD_BF16 ? 1 : 0;
    const GuardSpan spans[kGuardTensors] = {
        {a.x, b * L * h * p, io16}, {a.dt, b * L * h, 0},     {a.dt_bias, h, 0},  {a.A, h, 0},
        {a.B, b * L * gr * n, io16}, {a.C, b * L * gr * n, io16}, {a.D, h, 0}, {a.init, b * h * p * n, 0},
    };
    long long most = 0;
    for (int i = 0; i < kGuardTensors; ++i) {
        g.s[i] = spans[i];
        if (spans[i].p) most = std::max(most, spans[i].n);
    }
    cudaStream_t s = a.stream;
    unsigned long long* dcounts = nullptr;
    if (cudaMallocAsync(reinterpret_cast<void**>(&dcounts), sizeof(unsigned long long) * kGuardTensors, s) !=
        cudaSuccess)
        return SSD_ERR_CUDA;
    g.counts = dcounts;
    unsigned long long host[kGuardTensors] = {};
    bool ok = cudaMemsetAsync(dcounts, 0, sizeof(host), s) == cudaSuccess;
    if (ok) {
        int dev = 0, nsm = 0;
        ok = cudaGetDevice(&dev) == cudaSuccess &&
             cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && nsm > 0;
        // enough blocks for the largest tensor's 16-byte loads, at most 4 per SM per tensor
        const long long want = (most / 4 + kGuardThreads - 1) / kGuardThreads;
        const unsigned gx = static_cast<unsigned>(std::max(1LL, std::min(want, 4LL * nsm)));
        if (ok) {
            count_nonfinite<<<dim3(gx, kGuardTensors), kGuardThreads, 0, s>>>(g);
            note_launches(1);
            ok = cudaGetLastError() == cudaSuccess;
        }
    }
    if (ok) ok = cudaMemcpyAsync(host, dcounts, sizeof(host), cudaMemcpyDeviceToHost, s) == cudaSuccess;
    const bool freed = cudaFreeAsync(dcounts, s) == cudaSuccess;
    if (!ok || !freed || cudaStreamSynchronize(s) != cudaSuccess) return SSD_ERR_CUDA;
    for (int i = 0; i < kGuardTensors; ++i) counts[i] = static_cast<int64_t>(host[i]);
    return SSD_OK;
}

}  // namespace ssd
