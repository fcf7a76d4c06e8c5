// The C ABI of libssd (include/ssd.h): argument checks, path selection,
// library-owned workspaces and staging buffers, the device status word.
#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "ssd_internal.h"

namespace ssd {
namespace {

std::atomic<uint64_t> g_launches{0};

// Word 0: bit 0 / 1: a bounded device-side wait gave up (see the kernels);
// bit 3: a debug-build index check failed (SSD_CHECK). Word 1: source line of
// the first failed debug check.
__device__ unsigned g_status_word[2];

constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s per device-side wait
constexpr int kMaxDevices = 64;
constexpr int kHostSlices = 16;           // ssd_fwd_host: token slices in the upload / forward / download pipeline, at most
constexpr int kHostMinSlices = 4;         // ssd_fwd_host: at least, where the sequence allows
constexpr int64_t kHostSliceBytes = 96ll << 20;  // ssd_fwd_host: copy bytes per slice above kHostMinSlices slices
constexpr int64_t kHostSliceMinTokens = 512;  // ssd_fwd_host: no slice shorter (unless the sequence is)
constexpr int64_t kHostCutAlign = 256;        // ssd_fwd_host: cuts on multiples of this many tokens

struct DeviceState {
    unsigned* status = nullptr;     // device address of g_status_word
    void* ws = nullptr;             // library-owned workspace
    size_t ws_bytes = 0;
    // staging for ssd_fwd_host: device copies of the inputs and outputs, one
    // workspace (the slices' forwards run one after another), three streams
    // (uploads, forwards, downloads) and the events that order them
    void* dev_io = nullptr;
    size_t dev_io_bytes = 0;
    cudaStream_t host_stream[3] = {};
    cudaEvent_t host_event[2 * kHostSlices + 2] = {};
    void* slice_ws = nullptr;
    size_t slice_ws_bytes = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Limit on a kernel's wait for state published by another CTA. The
// environment variable SSD_DEVICE_WAIT_NS (read at every call) overrides it;
// tests shrink it to exercise the timeout path.
unsigned long long wait_limit_ns() {
    const char* e = std::getenv("SSD_DEVICE_WAIT_NS");
    if (e && *e) {
        const unsigned long long x = std::strtoull(e, nullptr, 10);
        if (x > 0) return x;
    }
    return kDefaultWaitNs;
}

// ssd_fwd_host's slice count before the caps of the sequence length: the
// environment variable SSD_HOST_SLICES (read at every call, 1 .. kHostSlices)
// overrides the rule from the copy bytes; tests use it to force many slices on
// small inputs.
int64_t host_slices_wanted(int64_t copy_bytes) {
    const char* e = std::getenv("SSD_HOST_SLICES");
    if (e && *e) {
        const long v = std::strtol(e, nullptr, 10);
        if (v >= 1 && v <= kHostSlices) return v;
    }
    return std::max<int64_t>(kHostMinSlices, (copy_bytes + kHostSliceBytes - 1) / kHostSliceBytes);
}

// Chain path warm-up mode (FwdArgs::chain_warmup). The environment variable
// SSD_CHAIN_WARMUP (read at every call: 0, 1 or 2) overrides the default 1;
// tests use 0 to force the hand-off path and 2 to force warm-ups.
int chain_warmup_mode() {
    const char* e = std::getenv("SSD_CHAIN_WARMUP");
    if (e && (e[0] == '0' || e[0] == '1' || e[0] == '2') && e[1] == '\0') return e[0] - '0';
    return 1;
}

ssd_status current_device(int* dev) {
    if (cudaGetDevice(dev) != cudaSuccess) return SSD_ERR_CUDA;
    if (*dev < 0 || *dev >= kMaxDevices) return SSD_ERR_UNSUPPORTED;
    return SSD_OK;
}

// Device address of the status word for the current device (cached).
ssd_status status_word(int dev, unsigned** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& s = g_dev[dev];
    if (!s.status) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return SSD_ERR_CUDA;
        s.status = static_cast<unsigned*>(p);
    }
    *out = s.status;
    return SSD_OK;
}

ssd_status check_dims(const ssd_dims* d, ssd_dtype io, int chunk_len, int ngroups) {
    if (!d) return SSD_ERR_INVALID_ARG;
    if (d->batch < 1 || d->seqlen < 1 || d->nheads < 1 || d->headdim < 1 || d->ngroups < 1 || d->dstate < 1)
        return SSD_ERR_INVALID_ARG;
    if (d->nheads % d->ngroups != 0) return SSD_ERR_INVALID_ARG;
    if (ngroups != d->ngroups) return SSD_ERR_INVALID_ARG;
    if (io != SSD_F32 && io != SSD_BF16) return SSD_ERR_INVALID_ARG;
    if (chunk_len < 1) return SSD_ERR_INVALID_ARG;
    return SSD_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ssd_status check_pointers(const void* x, const float* dt, const float* dt_bias, const float* A, const void* B,
                          const void* C, const float* D, const float* init, const void* y, const float* fs) {
    if (!x || !dt || !dt_bias || !A || !B || !C || !y) return SSD_ERR_INVALID_ARG;
    for (const void* p : {x, static_cast<const void*>(dt), static_cast<const void*>(dt_bias),
                          static_cast<const void*>(A), B, C, y})
        if (!aligned16(p)) return SSD_ERR_UNSUPPORTED;
    for (const void* p : {static_cast<const void*>(D), static_cast<const void*>(init), static_cast<const void*>(fs)})
        if (p && !aligned16(p)) return SSD_ERR_UNSUPPORTED;
    return SSD_OK;
}

ssd_path resolve_path(const ssd_dims& d, ssd_dtype io, int chunk_len, ssd_path want) {
    if (want != SSD_PATH_AUTO) return want;
    if (chain_supported(d, io, chunk_len)) return SSD_PATH_CHAIN;
    if (tc_supported(d, io, chunk_len)) return SSD_PATH_TC;
    return SSD_PATH_SIMT;
}

bool path_supported(const ssd_dims& d, ssd_dtype io, int chunk_len, ssd_path path) {
    if (path == SSD_PATH_TC) return tc_supported(d, io, chunk_len);
    if (path == SSD_PATH_CHAIN) return chain_supported(d, io, chunk_len);
    if (path == SSD_PATH_SIMT) return simt_supported(d, chunk_len);
    return false;
}

size_t workspace_for(const ssd_dims& d, int chunk_len, ssd_path path) {
    if (path == SSD_PATH_TC) return tc_workspace_bytes(d, chunk_len);
    if (path == SSD_PATH_CHAIN) return chain_workspace_bytes(d);
    return simt_workspace_bytes(d, chunk_len);
}

ssd_status run(const ssd_dims* dims, ssd_dtype io, const void* x, const float* dt, const float* dt_bias,
               const float* A, const void* B, const void* C, const float* D, const float* init, int chunk_len,
               int ngroups, void* y, float* fs, ssd_path path, void* ws, size_t ws_bytes, bool own_ws,
               void* stream, float dt_min = 0.f, float dt_max = __builtin_inff(),
               const int32_t* seq_idx = nullptr) {
    ssd_status st = check_dims(dims, io, chunk_len, ngroups);
    if (st != SSD_OK) return st;
    if (path != SSD_PATH_AUTO && path != SSD_PATH_SIMT && path != SSD_PATH_TC && path != SSD_PATH_CHAIN)
        return SSD_ERR_INVALID_ARG;
    st = check_pointers(x, dt, dt_bias, A, B, C, D, init, y, fs);
    if (st != SSD_OK) return st;
    if (seq_idx && (reinterpret_cast<uintptr_t>(seq_idx) & 3u) != 0) return SSD_ERR_UNSUPPORTED;
    const ssd_path p = resolve_path(*dims, io, chunk_len, path);
    if (!path_supported(*dims, io, chunk_len, p)) return SSD_ERR_UNSUPPORTED;
    const size_t need = workspace_for(*dims, chunk_len, p);
    if (!own_ws &&
        (ws_bytes < need || (need > 0 && !ws) || (reinterpret_cast<uintptr_t>(ws) % kWorkspaceAlign) != 0))
        return SSD_ERR_WORKSPACE;

    int dev = 0;
    st = current_device(&dev);
    if (st != SSD_OK) return st;
    unsigned* status = nullptr;
    st = status_word(dev, &status);
    if (st != SSD_OK) return st;

    if (own_ws) {
        std::lock_guard<std::mutex> lock(g_mu);
        DeviceState& s = g_dev[dev];
        if (s.ws_bytes < need) {
            if (s.ws) {
                // a smaller workspace may still be in use by work queued earlier
                if (cudaDeviceSynchronize() != cudaSuccess) return SSD_ERR_CUDA;
                cudaFree(s.ws);
                s.ws = nullptr;
                s.ws_bytes = 0;
            }
            if (cudaMalloc(&s.ws, need) != cudaSuccess) return SSD_ERR_CUDA;
            // the tensor-core path's state slots must start zero-filled (see ssd_fwd_ws)
            if (cudaMemset(s.ws, 0, need) != cudaSuccess) return SSD_ERR_CUDA;
            s.ws_bytes = need;
        }
        ws = s.ws;
        ws_bytes = s.ws_bytes;
    }

    FwdArgs a;
    a.d = *dims;
    a.io = io;
    a.x = x;
    a.dt = dt;
    a.dt_bias = dt_bias;
    a.A = A;
    a.B = B;
    a.C = C;
    a.D = D;
    a.init = init;
    a.chunk_len = chunk_len;
    a.y = y;
    a.final_state = fs;
    a.stream = static_cast<cudaStream_t>(stream);
    a.status_word = status;
    a.wait_limit_ns = wait_limit_ns();
    a.dt_min = dt_min;
    a.dt_max = dt_max;
    a.chain_warmup = chain_warmup_mode();
    a.seq_idx = seq_idx;
    if (p == SSD_PATH_TC) return tc_forward(a, ws, ws_bytes);
    if (p == SSD_PATH_CHAIN) return chain_forward(a, ws, ws_bytes);
    return simt_forward(a, ws, ws_bytes);
}

size_t elem_bytes(ssd_dtype io) { return io == SSD_F32 ? 4 : 2; }

// Token slices of ssd_fwd_host for valid dims: one per kHostSliceBytes of
// copies, at least kHostMinSlices (fewer slices leave the link idle in one
// direction for longer at both ends, more pay each forward's fixed cost more
// often), at most kHostSlices, none shorter than kHostSliceMinTokens.
int host_slice_count(const ssd_dims& d, ssd_dtype io) {
    const int64_t eb = static_cast<int64_t>(elem_bytes(io));
    const int64_t per_token = 2 * eb * d.nheads * d.headdim + 4 * d.nheads + 2 * eb * d.ngroups * d.dstate;
    const int64_t copy_bytes = per_token * d.seqlen * d.batch;
    return static_cast<int>(std::max<int64_t>(
        1, std::min<int64_t>({static_cast<int64_t>(kHostSlices), d.seqlen / kHostSliceMinTokens,
                              host_slices_wanted(copy_bytes)})));
}

// A dt limit is 0 <= dt_min <= dt_max (dt_max may be +inf); NULL means none.
bool dt_limit_ok(const ssd_dt_limit* lim, float* lo, float* hi) {
    *lo = 0.f;
    *hi = __builtin_inff();
    if (!lim) return true;
    if (!(lim->dt_min >= 0.f) || !(lim->dt_max >= lim->dt_min)) return false;  // also rejects NaN
    *lo = lim->dt_min;
    *hi = lim->dt_max;
    return true;
}

// ---- fixed scratch for ssd_fwd_noalloc
// Some callers must not allocate device memory (see ssd_fwd_noalloc in
// ssd.h), so that entry point runs the fused kernel on this file-scope array
// instead of the library-owned workspace. It is part of the loaded module:
// every device that loads the library holds these bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the fixed scratch on device `dev` (which must be current).
// The first call per device looks the address up and zero-fills the array
// once; both are synchronous, which is why the first ssd_fwd_noalloc call on a
// device belongs before any stream capture.
ssd_status noalloc_scratch(int dev, void** out) {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SSD_ERR_CUDA;
        if (cudaMemset(p, 0, kNoAllocScratchBytes) != cudaSuccess) return SSD_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess) return SSD_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return SSD_OK;
}

}  // namespace

void note_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

// ---- ssd_kernel_timing
std::atomic<int> g_timing{0};
std::mutex g_timing_mu;
std::vector<std::pair<cudaEvent_t, cudaEvent_t>> g_timed;  // recorded pairs, not yet read
std::vector<cudaEvent_t> g_spare_events;
thread_local cudaEvent_t t_begin = nullptr;  // begin event of the launch this host thread is timing

cudaEvent_t timing_event() {
    std::lock_guard<std::mutex> lock(g_timing_mu);
    if (!g_spare_events.empty()) {
        cudaEvent_t e = g_spare_events.back();
        g_spare_events.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

void timing_begin(cudaStream_t s) {
    if (!g_timing.load(std::memory_order_relaxed)) return;
    t_begin = timing_event();
    if (t_begin && cudaEventRecord(t_begin, s) != cudaSuccess) t_begin = nullptr;
}

void timing_end(cudaStream_t s) {
    if (!t_begin) return;
    cudaEvent_t e = timing_event();
    if (e && cudaEventRecord(e, s) == cudaSuccess) {
        std::lock_guard<std::mutex> lock(g_timing_mu);
        g_timed.emplace_back(t_begin, e);
    }
    t_begin = nullptr;
}

}  // namespace ssd

using namespace ssd;

extern "C" {

ssd_status ssd_fwd(const ssd_dims* dims, ssd_dtype io_dtype, const void* x, const float* dt, const float* dt_bias,
                   const float* A, const void* B, const void* C, const float* D, const float* init_state,
                   int chunk_len, int ngroups, void* y, float* final_state, void* stream) {
    return run(dims, io_dtype, x, dt, dt_bias, A, B, C, D, init_state, chunk_len, ngroups, y, final_state,
               SSD_PATH_AUTO, nullptr, 0, true, stream);
}

ssd_status ssd_fwd_ws(const ssd_dims* dims, ssd_dtype io_dtype, const void* x, const float* dt,
                      const float* dt_bias, const float* A, const void* B, const void* C, const float* D,
                      const float* init_state, int chunk_len, int ngroups, void* y, float* final_state,
                      ssd_path path, void* workspace, size_t workspace_bytes, void* stream) {
    return run(dims, io_dtype, x, dt, dt_bias, A, B, C, D, init_state, chunk_len, ngroups, y, final_state, path,
               workspace, workspace_bytes, false, stream);
}

ssd_status ssd_fwd_ex(const ssd_dims* dims, ssd_dtype io_dtype, const void* x, const float* dt,
                      const float* dt_bias, const float* A, const void* B, const void* C, const float* D,
                      const float* init_state, int chunk_len, int ngroups, void* y, float* final_state,
                      const ssd_dt_limit* dt_limit, const int32_t* seq_idx, ssd_path path, void* workspace,
                      size_t workspace_bytes, void* stream) {
    float lo, hi;
    if (!dt_limit_ok(dt_limit, &lo, &hi)) return SSD_ERR_INVALID_ARG;
    const bool own = workspace == nullptr;
    return run(dims, io_dtype, x, dt, dt_bias, A, B, C, D, init_state, chunk_len, ngroups, y, final_state, path,
               workspace, workspace_bytes, own, stream, lo, hi, seq_idx);
}

size_t ssd_fwd_workspace_bytes(const ssd_dims* dims, ssd_dtype io_dtype, int chunk_len, ssd_path path) {
    if (check_dims(dims, io_dtype, chunk_len, dims ? static_cast<int>(dims->ngroups) : 0) != SSD_OK) return 0;
    if (path != SSD_PATH_AUTO && path != SSD_PATH_SIMT && path != SSD_PATH_TC && path != SSD_PATH_CHAIN) return 0;
    const ssd_path p = resolve_path(*dims, io_dtype, chunk_len, path);
    if (!path_supported(*dims, io_dtype, chunk_len, p)) return 0;
    return workspace_for(*dims, chunk_len, p);
}

int ssd_host_slices(const ssd_dims* dims, ssd_dtype io_dtype) {
    if (!dims || check_dims(dims, io_dtype, 1, static_cast<int>(dims->ngroups)) != SSD_OK) return 0;
    return host_slice_count(*dims, io_dtype);
}

ssd_path ssd_select_path(const ssd_dims* dims, ssd_dtype io_dtype, int chunk_len) {
    if (!dims) return SSD_PATH_SIMT;
    return resolve_path(*dims, io_dtype, chunk_len, SSD_PATH_AUTO);
}

ssd_status ssd_fwd_host(const ssd_dims* dims, ssd_dtype io_dtype, const void* x, const float* dt,
                        const float* dt_bias, const float* A, const void* B, const void* C, const float* D,
                        const float* init_state, int chunk_len, int ngroups, void* y, float* final_state,
                        void* stream) {
    ssd_status st = check_dims(dims, io_dtype, chunk_len, ngroups);
    if (st != SSD_OK) return st;
    if (!x || !dt || !dt_bias || !A || !B || !C || !y) return SSD_ERR_INVALID_ARG;
    const ssd_dims& d = *dims;
    const size_t eb = elem_bytes(io_dtype);
    const size_t nb = static_cast<size_t>(d.batch), L = static_cast<size_t>(d.seqlen);
    // bytes per token of one batch row of each batched tensor, and one batch row's state
    const size_t tok_x = eb * d.nheads * d.headdim;
    const size_t tok_dt = 4 * d.nheads;
    const size_t tok_bc = eb * d.ngroups * d.dstate;
    const size_t row_state = 4 * d.nheads * d.headdim * d.dstate;
    const size_t sz_h = 4 * d.nheads;
    // device layout: x, y, dt, B, C (each holding slice after slice, a slice as
    // [batch, its tokens, ...]), dt_bias, A, D, the initial state, and two states
    // that pass from one slice's forward to the next
    const size_t sizes[10] = {tok_x * L * nb, tok_x * L * nb, tok_dt * L * nb, tok_bc * L * nb, tok_bc * L * nb,
                              sz_h, sz_h, sz_h, row_state * nb, 2 * row_state * nb};
    size_t offs[10], total = 0;
    for (int i = 0; i < 10; ++i) {
        offs[i] = total;
        total += align_up(sizes[i], kWorkspaceAlign);
    }
    // The sequence is cut into token slices of all batch rows; each slice's
    // final state is the next one's initial state, which is exact for any cut
    // (the state carries everything before it). The upload of one slice, the
    // forward of another and the download of a third overlap, while every
    // forward still covers the whole batch. Each of the three steps has a stream
    // of its own and takes the slices in order. Cuts fall on whole multiples of
    // kHostCutAlign tokens (whole chunks and blocks of the tensor-core paths).
    const int nsl = host_slice_count(d, io_dtype);
    int64_t cut[kHostSlices + 1];
    cut[0] = 0;
    cut[nsl] = d.seqlen;
    for (int i = 1; i < nsl; ++i) {
        const int64_t c = d.seqlen * i / nsl;  // at least kHostSliceMinTokens past the previous cut
        cut[i] = c / kHostCutAlign * kHostCutAlign;
    }
    size_t ws_need = 0;
    for (int i = 0; i < nsl; ++i) {
        ssd_dims ds = d;
        ds.seqlen = cut[i + 1] - cut[i];
        const ssd_path p = resolve_path(ds, io_dtype, chunk_len, SSD_PATH_AUTO);
        if (!path_supported(ds, io_dtype, chunk_len, p)) return SSD_ERR_UNSUPPORTED;
        ws_need = std::max(ws_need, align_up(workspace_for(ds, chunk_len, p), kWorkspaceAlign));
    }
    int dev = 0;
    st = current_device(&dev);
    if (st != SSD_OK) return st;
    int max_pitch = 0;
    if (cudaDeviceGetAttribute(&max_pitch, cudaDevAttrMaxPitch, dev) != cudaSuccess) return SSD_ERR_CUDA;
    char* base = nullptr;
    char* wsb = nullptr;
    cudaStream_t up = nullptr, comp = nullptr, down = nullptr;
    cudaEvent_t ev[2 * kHostSlices + 2];
    {
        std::lock_guard<std::mutex> lock(g_mu);
        DeviceState& s = g_dev[dev];
        if (s.dev_io_bytes < total || s.slice_ws_bytes < ws_need) {
            if (cudaDeviceSynchronize() != cudaSuccess) return SSD_ERR_CUDA;  // the old buffers may be in use
            if (s.dev_io_bytes < total) {
                if (s.dev_io) cudaFree(s.dev_io);
                s.dev_io = nullptr;
                s.dev_io_bytes = 0;
                if (cudaMalloc(&s.dev_io, total) != cudaSuccess) return SSD_ERR_CUDA;
                s.dev_io_bytes = total;
            }
            if (s.slice_ws_bytes < ws_need) {
                if (s.slice_ws) cudaFree(s.slice_ws);
                s.slice_ws = nullptr;
                s.slice_ws_bytes = 0;
                if (cudaMalloc(&s.slice_ws, ws_need) != cudaSuccess) return SSD_ERR_CUDA;
                // the tensor-core path's state slots must start zero-filled (see ssd_fwd_ws)
                if (cudaMemset(s.slice_ws, 0, ws_need) != cudaSuccess) return SSD_ERR_CUDA;
                s.slice_ws_bytes = ws_need;
            }
        }
        for (cudaStream_t& hs : s.host_stream)
            if (!hs && cudaStreamCreateWithFlags(&hs, cudaStreamNonBlocking) != cudaSuccess) return SSD_ERR_CUDA;
        for (cudaEvent_t& he : s.host_event)
            if (!he && cudaEventCreateWithFlags(&he, cudaEventDisableTiming) != cudaSuccess) return SSD_ERR_CUDA;
        base = static_cast<char*>(s.dev_io);
        wsb = static_cast<char*>(s.slice_ws);
        up = s.host_stream[0];
        comp = s.host_stream[1];
        down = s.host_stream[2];
        for (int i = 0; i < 2 * kHostSlices + 2; ++i) ev[i] = s.host_event[i];
        ws_need = s.slice_ws_bytes;
    }
    cudaStream_t user = static_cast<cudaStream_t>(stream);
    auto cp = [](void* dst, const void* src, size_t n, cudaMemcpyKind k, cudaStream_t st_) {
        return n == 0 || cudaMemcpyAsync(dst, src, n, k, st_) == cudaSuccess;
    };
    // a slice of every batch row in one 2-D copy: nb rows of `width` bytes,
    // `spitch` apart in the source and `dpitch` apart in the destination (row by
    // row where a pitch is beyond what a 2-D copy takes)
    auto cp2 = [&](void* dst, size_t dpitch, const void* src, size_t spitch, size_t width, cudaMemcpyKind k,
                   cudaStream_t st_) {
        if (width == 0) return true;
        if (dpitch <= static_cast<size_t>(max_pitch) && spitch <= static_cast<size_t>(max_pitch))
            return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, nb, k, st_) == cudaSuccess;
        for (size_t r = 0; r < nb; ++r)
            if (cudaMemcpyAsync(static_cast<char*>(dst) + r * dpitch, static_cast<const char*>(src) + r * spitch, width,
                                k, st_) != cudaSuccess)
                return false;
        return true;
    };
    // on a failure after work was queued, nothing may still use the staging buffers on return
    auto fail = [&](ssd_status e) {
        for (cudaStream_t t : {up, comp, down, user}) cudaStreamSynchronize(t);
        return e;
    };
    // events: uploaded[i], computed[i], the per-head parameters, all downloads done
    cudaEvent_t* uploaded = ev;
    cudaEvent_t* computed = ev + kHostSlices;
    cudaEvent_t params = ev[2 * kHostSlices], done = ev[2 * kHostSlices + 1];
    // the per-head parameters go first on the caller's stream; the pipeline waits for them
    // (and so for everything the caller queued before)
    if (!cp(base + offs[5], dt_bias, sz_h, cudaMemcpyHostToDevice, user) ||
        !cp(base + offs[6], A, sz_h, cudaMemcpyHostToDevice, user) ||
        (D && !cp(base + offs[7], D, sz_h, cudaMemcpyHostToDevice, user)))
        return fail(SSD_ERR_CUDA);
    if (cudaEventRecord(params, user) != cudaSuccess || cudaStreamWaitEvent(up, params, 0) != cudaSuccess ||
        cudaStreamWaitEvent(comp, params, 0) != cudaSuccess || cudaStreamWaitEvent(down, params, 0) != cudaSuccess)
        return fail(SSD_ERR_CUDA);
    const char* hx = static_cast<const char*>(x);
    const char* hdt = reinterpret_cast<const char*>(dt);
    const char* hB = static_cast<const char*>(B);
    const char* hC = static_cast<const char*>(C);
    char* hy = static_cast<char*>(y);
    char* dinit = base + offs[8];
    float* pass[2] = {reinterpret_cast<float*>(base + offs[9]), reinterpret_cast<float*>(base + offs[9] + row_state * nb)};
    if (init_state && !cp(dinit, init_state, row_state * nb, cudaMemcpyHostToDevice, up)) return fail(SSD_ERR_CUDA);
    for (int i = 0; i < nsl; ++i) {
        const size_t l0 = static_cast<size_t>(cut[i]), ls = static_cast<size_t>(cut[i + 1] - cut[i]);
        // slice i of each batched tensor sits after slices 0 .. i-1, which hold l0 tokens of every row
        char* dx = base + offs[0] + tok_x * nb * l0;
        char* dy = base + offs[1] + tok_x * nb * l0;
        char* ddt = base + offs[2] + tok_dt * nb * l0;
        char* dB = base + offs[3] + tok_bc * nb * l0;
        char* dC = base + offs[4] + tok_bc * nb * l0;
        if (!cp2(dx, tok_x * ls, hx + tok_x * l0, tok_x * L, tok_x * ls, cudaMemcpyHostToDevice, up) ||
            !cp2(ddt, tok_dt * ls, hdt + tok_dt * l0, tok_dt * L, tok_dt * ls, cudaMemcpyHostToDevice, up) ||
            !cp2(dB, tok_bc * ls, hB + tok_bc * l0, tok_bc * L, tok_bc * ls, cudaMemcpyHostToDevice, up) ||
            !cp2(dC, tok_bc * ls, hC + tok_bc * l0, tok_bc * L, tok_bc * ls, cudaMemcpyHostToDevice, up) ||
            cudaEventRecord(uploaded[i], up) != cudaSuccess || cudaStreamWaitEvent(comp, uploaded[i], 0) != cudaSuccess)
            return fail(SSD_ERR_CUDA);
        ssd_dims ds = d;
        ds.seqlen = static_cast<int64_t>(ls);
        const float* init = i > 0 ? pass[(i - 1) & 1] : (init_state ? reinterpret_cast<const float*>(dinit) : nullptr);
        float* fin = (i + 1 < nsl || final_state) ? pass[i & 1] : nullptr;
        st = run(&ds, io_dtype, dx, reinterpret_cast<const float*>(ddt),
                 reinterpret_cast<const float*>(base + offs[5]), reinterpret_cast<const float*>(base + offs[6]), dB,
                 dC, D ? reinterpret_cast<const float*>(base + offs[7]) : nullptr, init, chunk_len, ngroups, dy, fin,
                 SSD_PATH_AUTO, wsb, ws_need, false, comp);
        if (st != SSD_OK) return fail(st);
        if (cudaEventRecord(computed[i], comp) != cudaSuccess || cudaStreamWaitEvent(down, computed[i], 0) != cudaSuccess)
            return fail(SSD_ERR_CUDA);
        if (!cp2(hy + tok_x * l0, tok_x * L, dy, tok_x * ls, tok_x * ls, cudaMemcpyDeviceToHost, down))
            return fail(SSD_ERR_CUDA);
    }
    if (final_state && !cp(final_state, pass[(nsl - 1) & 1], row_state * nb, cudaMemcpyDeviceToHost, down))
        return fail(SSD_ERR_CUDA);
    if (cudaEventRecord(done, down) != cudaSuccess || cudaStreamWaitEvent(user, done, 0) != cudaSuccess)
        return fail(SSD_ERR_CUDA);
    return ssd_device_status(stream);
}

ssd_status ssd_check_inputs(const ssd_dims* dims, ssd_dtype io_dtype, const void* x, const float* dt,
                            const float* dt_bias, const float* A, const void* B, const void* C, const float* D,
                            const float* init_state, int64_t* counts, void* stream) {
    if (!dims || !counts) return SSD_ERR_INVALID_ARG;
    const ssd_status st = check_dims(dims, io_dtype, 1, static_cast<int>(dims->ngroups));
    if (st != SSD_OK) return st;
    if (!x || !dt || !dt_bias || !A || !B || !C) return SSD_ERR_INVALID_ARG;
    const uintptr_t io_size = io_dtype == SSD_BF16 ? 2 : 4;
    for (const void* p : {x, B, C})
        if (reinterpret_cast<uintptr_t>(p) % io_size != 0) return SSD_ERR_UNSUPPORTED;
    for (const float* p : {dt, dt_bias, A, D, init_state})
        if (p && reinterpret_cast<uintptr_t>(p) % 4 != 0) return SSD_ERR_UNSUPPORTED;
    const CheckArgs a{*dims, io_dtype, x, dt, dt_bias, A, B, C, D, init_state, static_cast<cudaStream_t>(stream)};
    return check_inputs(a, counts);
}

ssd_status ssd_device_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SSD_ERR_CUDA;
    int dev = 0;
    ssd_status st = current_device(&dev);
    if (st != SSD_OK) return st;
    unsigned* word = nullptr;
    st = status_word(dev, &word);
    if (st != SSD_OK) return st;
    unsigned v = 0;
    if (cudaMemcpy(&v, word, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return SSD_ERR_CUDA;
    if (v != 0) {
        const unsigned zero[2] = {0, 0};
        if (cudaMemcpy(word, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return SSD_ERR_CUDA;
        return (v & 8u) ? SSD_ERR_DEBUG_CHECK : SSD_ERR_DEVICE_TIMEOUT;
    }
    return SSD_OK;
}

const char* ssd_status_string(ssd_status status) {
    switch (status) {
        case SSD_OK: return "ok";
        case SSD_ERR_INVALID_ARG: return "invalid argument";
        case SSD_ERR_UNSUPPORTED: return "unsupported shape, dtype, chunk length or alignment";
        case SSD_ERR_CUDA: return "CUDA error";
        case SSD_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        case SSD_ERR_WORKSPACE: return "workspace too small or misaligned";
        case SSD_ERR_DEBUG_CHECK: return "a debug-build index or bounds check failed in a kernel";
    }
    return "unknown status";
}

uint64_t ssd_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int ssd_debug_build(void) {
#ifdef SSD_DEBUG
    return 1;
#else
    return 0;
#endif
}

unsigned ssd_debug_failed_line(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return 0;
    int dev = 0;
    if (current_device(&dev) != SSD_OK) return 0;
    unsigned* word = nullptr;
    if (status_word(dev, &word) != SSD_OK) return 0;
    unsigned v[2] = {0, 0};
    if (cudaMemcpy(v, word, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return 0;
    return v[1];
}

void ssd_kernel_timing(int enable) { g_timing.store(enable ? 1 : 0, std::memory_order_relaxed); }

ssd_status ssd_kernel_timing_read(double* total_ms, uint64_t* count) {
    if (!total_ms || !count) return SSD_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_timing_mu);
    double sum = 0.0;
    ssd_status st = SSD_OK;
    for (auto& pr : g_timed) {
        float ms = 0.f;
        if (cudaEventSynchronize(pr.second) != cudaSuccess || cudaEventElapsedTime(&ms, pr.first, pr.second) != cudaSuccess)
            st = SSD_ERR_CUDA;
        sum += ms;
        g_spare_events.push_back(pr.first);
        g_spare_events.push_back(pr.second);
    }
    *total_ms = sum;
    *count = g_timed.size();
    g_timed.clear();
    return st;
}

void ssd_release(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    int prev = 0;
    const bool have_prev = cudaGetDevice(&prev) == cudaSuccess;
    for (int d = 0; d < kMaxDevices; ++d) {
        DeviceState& s = g_dev[d];
        if (!s.ws && !s.dev_io && !s.slice_ws && !s.host_stream[0]) continue;
        if (cudaSetDevice(d) != cudaSuccess) continue;
        cudaDeviceSynchronize();
        if (s.ws) cudaFree(s.ws);
        if (s.dev_io) cudaFree(s.dev_io);
        if (s.slice_ws) cudaFree(s.slice_ws);
        for (cudaStream_t& hs : s.host_stream)
            if (hs) cudaStreamDestroy(hs);
        for (cudaEvent_t& he : s.host_event)
            if (he) cudaEventDestroy(he);
        s = DeviceState{};
    }
    if (have_prev) cudaSetDevice(prev);
}


ssd_status ssd_fwd_noalloc(const ssd_dims* dims, ssd_dtype io_dtype, const void* x, const float* dt,
                           const float* dt_bias, const float* A, const void* B, const void* C, const float* D,
                           const float* init_state, int chunk_len, int ngroups, void* y, float* final_state,
                           void* stream) {
    ssd_status st = check_dims(dims, io_dtype, chunk_len, ngroups);
    if (st != SSD_OK) return st;
    st = check_pointers(x, dt, dt_bias, A, B, C, D, init_state, y, final_state);
    if (st != SSD_OK) return st;
    if (!tc_supported(*dims, io_dtype, chunk_len)) return SSD_ERR_UNSUPPORTED;
    if (tc_workspace_bytes(*dims, chunk_len) > kNoAllocScratchBytes) return SSD_ERR_WORKSPACE;
    int dev = 0;
    st = current_device(&dev);
    if (st != SSD_OK) return st;
    unsigned* status = nullptr;
    st = status_word(dev, &status);
    if (st != SSD_OK) return st;
    void* scratch = nullptr;
    st = noalloc_scratch(dev, &scratch);
    if (st != SSD_OK) return st;
    FwdArgs a;
    a.d = *dims;
    a.io = io_dtype;
    a.x = x;
    a.dt = dt;
    a.dt_bias = dt_bias;
    a.A = A;
    a.B = B;
    a.C = C;
    a.D = D;
    a.init = init_state;
    a.chunk_len = chunk_len;
    a.y = y;
    a.final_state = final_state;
    a.stream = static_cast<cudaStream_t>(stream);
    a.status_word = status;
    a.wait_limit_ns = wait_limit_ns();
    return tc_forward(a, scratch, kNoAllocScratchBytes);
}

ssd_status ssd_step(const ssd_dims* dims, ssd_dtype io_dtype, const void* x, const float* dt, const float* dt_bias,
                    const float* A, const void* B, const void* C, const float* D, float* state, int ngroups, void* y,
                    void* stream) {
    return ssd_step_ex(dims, io_dtype, x, dt, dt_bias, A, B, C, D, state, ngroups, y, nullptr, stream);
}

ssd_status ssd_step_ex(const ssd_dims* dims, ssd_dtype io_dtype, const void* x, const float* dt,
                       const float* dt_bias, const float* A, const void* B, const void* C, const float* D,
                       float* state, int ngroups, void* y, const ssd_dt_limit* dt_limit, void* stream) {
    float lo, hi;
    if (!dt_limit_ok(dt_limit, &lo, &hi)) return SSD_ERR_INVALID_ARG;
    ssd_status st = check_dims(dims, io_dtype, 1, ngroups);
    if (st != SSD_OK) return st;
    if (dims->seqlen != 1) return SSD_ERR_INVALID_ARG;
    if (!state) return SSD_ERR_INVALID_ARG;
    st = check_pointers(x, dt, dt_bias, A, B, C, D, nullptr, y, state);
    if (st != SSD_OK) return st;
    if (!step_supported(*dims)) return SSD_ERR_UNSUPPORTED;
    int dev = 0;
    st = current_device(&dev);
    if (st != SSD_OK) return st;
    StepArgs a;
    a.d = *dims;
    a.io = io_dtype;
    a.x = x;
    a.dt = dt;
    a.dt_bias = dt_bias;
    a.A = A;
    a.B = B;
    a.C = C;
    a.D = D;
    a.state = state;
    a.y = y;
    a.stream = static_cast<cudaStream_t>(stream);
    a.dt_min = lo;
    a.dt_max = hi;
    return step_forward(a);
}

}  // extern "C"
