// Fused tcgen05/TMA path of the SSD forward (bf16 io, fp32 accumulation).
//
// Work unit: one 128-token block of one batch row for a group of up to 8
// heads that read the same B/C group. Units are handed out by an atomic
// ticket in block-major order (every batch row and head group of block k
// before any unit of block k+1), so a unit only ever waits on units that
// took their tickets earlier.
//
// Per unit the CTA loads B and C once and computes C.B^T once; its heads are
// then processed by SLOTS warpgroup pairs ("slots", 256 threads each) that
// take alternate heads, so one slot's waits overlap the other's work. Per
// head the five stages of the chunked SSD (burn-mamba "mamba2/ssd/serial.rs"
// k1..k5; fla "mamba2.py" naive chunked SSD) run as:
//
//   k1  dt = softplus(dt_raw + dt_bias), cs = inclusive cumsum of dt*A   (per unit, all heads)
//   k2  CB = C . B^T                 [128 x 128, K = dstate]   once per unit, tcgen05 -> TMEM
//   k3  S^T = B^T . diag(dt e^{cs_end-cs}) . X   [dstate x 64, K = 128]   tcgen05 -> TMEM
//   k5a Yd = (L o CB o dt + D I) . X [128 x 64, K = 128]       mask in registers, tcgen05
//   k4  s_out = e^{cs_end} s_in + S  fp32, chained through global slots (bounded waits)
//   k5b Yo = C . s_in^T              [128 x 64, K = dstate]    tcgen05
//       y  = e^{cs} o Yo + Yd        epilogue, TMA store
//
// The D skip rides on the diagonal of the masked matrix (D x_t = (D I) x).
// The decay e^{cs_t - cs_s} of row t is factored as u_t v_q(s) with
// u_t = e^{cs_t - cs_r}, v_q(s) = e^{cs_r - cs_s} dt_s and r the first row of
// t's 32-row quarter q, so the mask needs no per-entry exponential: the row
// factor u_t moves to the epilogue (and D to D/u_t on the diagonal). Quarters
// whose decay exceeds kMaxFactorLog keep exact entries instead.
// A chunk_len of 256 is computed as two consecutive 128-token blocks: the
// decomposition is exact for any chunk boundary, and the state between the
// two halves is passed through the same chained slots.
//
// Operand staging (128-byte swizzle throughout; see ptx.cuh):
//   sB [t][n]  (TMA, per unit)   B operand of k2 (K-major), A operand of k3 (MN-major)
//   sC [t][n]  (TMA, per unit)   A operand of k2 and k5b (K-major)
//   per slot:
//   sX [t][p]  (TMA, per head)   B operand of k5a (MN-major, K = t)
//   sW [t][p]  (threads)         dt e^{cs_end-cs} X, B operand of k3 (MN-major)
//   sM [t][s]  (threads)         masked CB, A operand of k5a (K-major)
//   sH [n][p]  (threads)         s_in in bf16, B operand of k5b (MN-major): in sW (dstate 128) or sM (256)
//   sY [t][p]  (threads)         y tile for the TMA store, in sW (after k5b has read sH)
#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>
#include <mutex>

#include "ptx.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kT = 128;               // tokens per block (MMA M for k2, k5a, k5b)
constexpr int kP = 64;                // headdim handled by this kernel
constexpr int kMaxHeads = 8;          // heads per unit at most
constexpr uint32_t kTile = kT * 128;  // one 128-row x 128-byte swizzled tile (16 KB)
constexpr uint32_t kPoison = 0xFFFFFFFFu;
// Limit on waits for this CTA's own TMA copies and MMAs (they complete in
// microseconds; the limit only guards against a wedged pipeline).
constexpr unsigned long long kLocalWaitNs = 2000000000ull;
// Largest decay (in nats) across a 32-row quarter for which the mask is stored
// in factored form; e^{60} * |D| stays far inside the bf16/fp32 range.
constexpr float kMaxFactorLog = 60.f;

template <int NST>
struct Cfg {
    static constexpr int NKB = NST / 64;                    // 64-wide dstate blocks
    static constexpr int SLOTS = (NST == 128) ? 2 : 1;
    static constexpr int THREADS = 256 * SLOTS;
    static constexpr uint32_t OFF_B = 0;
    static constexpr uint32_t OFF_C = OFF_B + NKB * kTile;
    static constexpr uint32_t OFF_SLOT = OFF_C + NKB * kTile;
    static constexpr uint32_t SLOT_BYTES = 4 * kTile;       // X, W, M (2 tiles)
    static constexpr uint32_t SX = 0, SW = kTile, SM = 2 * kTile;  // offsets inside a slot
    static constexpr uint32_t SH = (NST == 128) ? SW : SM;
    static constexpr uint32_t SY = SW;
    static constexpr uint32_t OFF_MISC = OFF_SLOT + SLOTS * SLOT_BYTES;
    // misc: 4 per-head tables [kMaxHeads][128] floats, per-slot v tables [4][128], scan totals
    static constexpr uint32_t TAB_BYTES = 4 * kMaxHeads * kT * 4;
    static constexpr uint32_t V_BYTES = SLOTS * 4 * kT * 4;
    static constexpr uint32_t MISC_BYTES = TAB_BYTES + V_BYTES + 512 + 256;
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + MISC_BYTES + 1024;  // + alignment slack
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_CB = 0;
    __host__ __device__ static constexpr uint32_t col_s(int slot) { return 128 + 128 * slot; }
    __host__ __device__ static constexpr uint32_t col_d(int slot) { return NST == 128 ? 192 + 128 * slot : 256; }
    __host__ __device__ static constexpr uint32_t col_o(int slot) { return col_s(slot); }
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(NST == 128 || SLOTS == 1, "one slot for dstate 256");
};

struct TcParams {
    const float* dt;
    const float* dt_bias;
    const float* A;
    const float* D;
    const float* init;
    float* final_state;
    uint64_t* slots;       // [batch*H][2][P/2][NST][2] chained states: fp32 value | tag << 32
    uint32_t* ticket;      // block-major work counter
    uint32_t epoch;        // per-call tag component
    uint32_t* status;      // device status word
    int batch, H, G, nblk, hpu, ngrp;  // hpu heads per unit, ngrp = H / hpu head groups
    long long L;
    unsigned long long chain_wait_ns;  // limit on waiting for the previous block's state
};

// Tag of the state block `blk` publishes in call `epoch`: never 0 (so zeroed
// memory never matches) and never kPoison, for blk < 65535.
__device__ __forceinline__ uint32_t state_tag(uint32_t epoch, int blk) {
    return ((epoch % 65535u + 1u) << 16) | static_cast<uint32_t>((blk + 1) & 0xFFFF);
}

__device__ __forceinline__ float softplus_f(float v) {
    return v > 0.f ? v + log1pf(expf(-v)) : log1pf(expf(v));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t v) {
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&v);
    return __bfloat1622float2(b);
}

// Bounded wait; a timeout is recorded in the status word (bit 1) and the
// caller proceeds (its results are then invalid, and the host is told).
__device__ __forceinline__ void wait_local(uint64_t* bar, uint32_t parity, uint32_t* status) {
    if (!ptx::mbar_wait(bar, parity, kLocalWaitNs)) atomicOr(status, 2u);
}

template <int NST>
__global__ void __launch_bounds__(Cfg<NST>::THREADS, 1)
    ssd_tc_fused(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
                 const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_y,
                 const TcParams prm) {
    using K = Cfg<NST>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* tCs = reinterpret_cast<float*>(smem + K::OFF_MISC);  // [head][t] inclusive cumsum of dt*A
    float* tDt = tCs + kMaxHeads * kT;                          // [head][t] dt
    float* tWt = tDt + kMaxHeads * kT;                          // [head][t] dt e^{cs_end - cs}
    float* tEt = tWt + kMaxHeads * kT;                          // [head][t] e^{cs}
    float* tV = tEt + kMaxHeads * kT;                           // [slot][q][s] e^{cs_{32q} - cs_s} dt_s
    float* tTot = tV + K::SLOTS * 4 * kT;                       // [head][4] scan totals
    float* tD = tTot + kMaxHeads * 4;                           // [head] D
    uint64_t* bars = reinterpret_cast<uint64_t*>(tTot + kMaxHeads * 4 + 32);
    static_assert(kMaxHeads * 4 + kMaxHeads <= kMaxHeads * 4 + 32, "tD fits before the barriers");
    // bars: [0] B/C, [1] CB, then per slot s: [2+4s] X, [3+4s] S, [4+4s] D, [5+4s] O
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(bars + 2 + 4 * K::SLOTS);
    int* sInfo = reinterpret_cast<int*>(sTmem + 1);             // [0] unit, [1+s] chain abort of slot s

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slot = tid >> 8, stid = tid & 255, swarp = stid >> 5;
    const int quarter = warp & 3, half = swarp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;

    if (tid == 0) {
        sInfo[0] = static_cast<int>(atomicAdd(prm.ticket, 1u));
#pragma unroll
        for (int i = 0; i < 2 + 4 * K::SLOTS; ++i) ptx::mbar_init(&bars[i], 1);
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(sTmem, K::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *sTmem;
    const int unit = sInfo[0];
    const int grp = unit % prm.ngrp;
    const int b = (unit / prm.ngrp) % prm.batch;
    const int blk = unit / (prm.ngrp * prm.batch);
    const int h0 = grp * prm.hpu;
    const int g = h0 / (prm.H / prm.G);
    const int t0 = blk * kT;
    const long long L = prm.L;
    const int hpu = prm.hpu;
    const uint32_t sbase = ptx::smem_u32(smem);
    uint8_t* slot_base = smem + K::OFF_SLOT + slot * K::SLOT_BYTES;
    const uint32_t slot_addr = sbase + K::OFF_SLOT + slot * K::SLOT_BYTES;
    uint64_t* bar_x = &bars[2 + 4 * slot];
    uint64_t* bar_s = &bars[3 + 4 * slot];
    uint64_t* bar_d = &bars[4 + 4 * slot];
    uint64_t* bar_o = &bars[5 + 4 * slot];
    const bool leader = (stid == 0);

    // ---- TMA: B and C for the unit; X for each slot's first head
    if (tid == 0) {
        ptx::mbar_arrive_expect_tx(&bars[0], 2 * K::NKB * kTile);
#pragma unroll
        for (int kb = 0; kb < K::NKB; ++kb) {
            ptx::tma_load_4d(smem + K::OFF_B + kb * kTile, &tm_b, &bars[0], 64 * kb, g, t0, b);
            ptx::tma_load_4d(smem + K::OFF_C + kb * kTile, &tm_c, &bars[0], 64 * kb, g, t0, b);
        }
    }
    if (leader && slot < hpu) {
        ptx::mbar_arrive_expect_tx(bar_x, kTile);
        ptx::tma_load_4d(slot_base + K::SX, &tm_x, bar_x, 0, h0 + slot, t0, b);
    }

    // ---- k1 for every head of the unit: dt, inclusive cumsum of dt*A (32-token warp scans)
    for (int task = warp; task < hpu * 4; task += K::THREADS / 32) {
        const int j = task >> 2, c4 = task & 3;
        const int h = h0 + j;
        const long long t = static_cast<long long>(t0) + 32 * c4 + lane;
        float dtv = 0.f;
        if (t < L) dtv = softplus_f(prm.dt[(static_cast<long long>(b) * L + t) * prm.H + h] + prm.dt_bias[h]);
        float v = dtv * prm.A[h];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += o;
        }
        tDt[j * kT + 32 * c4 + lane] = dtv;
        tCs[j * kT + 32 * c4 + lane] = v;
        if (lane == 31) tTot[j * 4 + c4] = v;
        if (c4 == 0 && lane == 0) tD[j] = prm.D ? prm.D[h] : 0.f;
    }
    __syncthreads();
    for (int e = tid; e < hpu * kT; e += K::THREADS) {
        const int j = e / kT, t = e % kT, c4 = t >> 5;
        float pre = 0.f;
        for (int c = 0; c < c4; ++c) pre += tTot[j * 4 + c];
        tCs[e] += pre;
    }
    __syncthreads();
    for (int e = tid; e < hpu * kT; e += K::THREADS) {
        const int j = e / kT;
        const float cs = tCs[e];
        const float cs_end = tCs[j * kT + kT - 1];
        tWt[e] = tDt[e] * __expf(cs_end - cs);
        tEt[e] = __expf(cs);
    }
    __syncthreads();

    // ---- k2: CB = C . B^T once per unit (M = t, N = s, K = n; both K-major)
    constexpr uint32_t IDESC_CB = ptx::idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t IDESC_S = ptx::idesc_bf16_f32(128, 64, true, true);
    constexpr uint32_t IDESC_D = ptx::idesc_bf16_f32(128, 64, false, true);
    constexpr uint32_t IDESC_O = ptx::idesc_bf16_f32(128, 64, false, true);
    if (tid == 0) {
        wait_local(&bars[0], 0, prm.status);
        ptx::tc_fence_after();
#pragma unroll
        for (int k = 0; k < NST / 16; ++k) {
            const uint32_t koff = (k >> 2) * kTile + (k & 3) * 32;
            const uint64_t da = ptx::desc_sw128(sbase + K::OFF_C + koff, 16, 1024);
            const uint64_t db = ptx::desc_sw128(sbase + K::OFF_B + koff, 16, 1024);
            ptx::mma_bf16(tmem + K::COL_CB, da, db, IDESC_CB, k > 0);
        }
        ptx::mma_commit(&bars[1]);
    }

    // Matrix descriptors are built once per issue from the operand base; a K
    // step adds its byte offset to the start-address field (offsets stay far
    // below the field's range).
    auto kmaj = [](int k) { return static_cast<uint64_t>(((k >> 2) * kTile + (k & 3) * 32) >> 4); };
    auto mnmaj = [](int k) { return static_cast<uint64_t>((k * 2048) >> 4); };

    // ---- per-slot head loop
    bool b_ready = false;  // this thread has seen B/C land
    int it = 0;
    for (int j = slot; j < hpu; j += K::SLOTS, ++it) {
        const int h = h0 + j;
        const uint32_t ph = it & 1;
        const float* cs = tCs + j * kT;
        const float* dts = tDt + j * kT;
        const float* wts = tWt + j * kT;
        float* vt = tV + slot * 4 * kT;
        // k4 bookkeeping for chain (b, h). Thread (quarter, half) owns state rows
        // n = 32*quarter + lane (+128 per tile) and columns p = 32*half .. +31.
        const int chain = b * prm.H + h;
        const uint64_t* prev = prm.slots + (static_cast<size_t>(chain) * 2 + ((blk - 1) & 1)) * kP * NST;
        uint64_t* mine = prm.slots + (static_cast<size_t>(chain) * 2 + (blk & 1)) * kP * NST;
        const uint32_t want = state_tag(prm.epoch, blk - 1);
        const uint32_t mine_tag = state_tag(prm.epoch, blk);
        const size_t fs_base = static_cast<size_t>(chain) * kP * NST;
        const int n0 = quarter * 32 + lane;
        // Slot layout [p/2][n][2] of 64-bit words: this thread's 32 words (rows
        // p = 32*half .. +31 of column n) come as 16 pairs of adjacent words.
        uint64_t w[32];
        auto load_words = [&](int mt) {
            const int n = n0 + 128 * mt;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                ptx::ld_relaxed_2xb64(prev + (static_cast<size_t>(16 * half + i) * NST + n) * 2, w[2 * i], w[2 * i + 1]);
        };

        // (a) the previous head's y store must have read its staging tile
        if (it > 0) {
            if (leader) ptx::bulk_wait_group_read0();
            ptx::named_sync(1 + slot, 256);
        }
        if (!b_ready) {
            wait_local(&bars[0], 0, prm.status);
            b_ready = true;
        }
        wait_local(bar_x, ph, prm.status);

        // (b) sW = X scaled by dt_t e^{cs_end - cs_t}; v table for the factored mask
#pragma unroll
        for (int i = 0; i < (kT * 8) / 256; ++i) {
            const int chunk = stid + i * 256;  // 16-byte chunk, 8 per 128-byte row
            const int row = chunk >> 3;
            const float w = wts[row];
            const uint4 v = *reinterpret_cast<const uint4*>(slot_base + K::SX + chunk * 16);
            const float2 f0 = unpack_bf16x2(v.x), f1 = unpack_bf16x2(v.y), f2 = unpack_bf16x2(v.z),
                         f3 = unpack_bf16x2(v.w);
            uint4 o;
            o.x = pack_bf16x2(f0.x * w, f0.y * w);
            o.y = pack_bf16x2(f1.x * w, f1.y * w);
            o.z = pack_bf16x2(f2.x * w, f2.y * w);
            o.w = pack_bf16x2(f3.x * w, f3.y * w);
            *reinterpret_cast<uint4*>(slot_base + K::SW + chunk * 16) = o;
        }
        // v_q(s) = e^{cs_{32q} - cs_s} dt_s for s < 32q + 32: 32 + 64 + 96 + 128 = 320 entries
        for (int idx = stid; idx < 320; idx += 256) {
            const int q = idx < 32 ? 0 : (idx < 96 ? 1 : (idx < 192 ? 2 : 3));
            const int s = idx - (q == 0 ? 0 : (q == 1 ? 32 : (q == 2 ? 96 : 192)));
            vt[q * kT + s] = __expf(fminf(cs[32 * q] - cs[s], kMaxFactorLog)) * dts[s];
        }
        ptx::fence_proxy_async_smem();
        ptx::named_sync(1 + slot, 256);

        // (c) k3: S^T = B^T . W  (M = n, N = p, K = t; both MN-major)
        if (leader) {
            ptx::tc_fence_after();
            const uint64_t dsc_b_mn = ptx::desc_sw128(sbase + K::OFF_B, kTile, 1024);  // B^T, MN-major
            const uint64_t dsc_w = ptx::desc_sw128(slot_addr + K::SW, kTile, 1024);   // W, MN-major
#pragma unroll
            for (int mt = 0; mt < NST / 128; ++mt) {
#pragma unroll
                for (int k = 0; k < kT / 16; ++k)
                    ptx::mma_bf16(tmem + K::col_s(slot) + 64 * mt, dsc_b_mn + ((2 * mt * kTile) >> 4) + mnmaj(k),
                                  dsc_w + mnmaj(k), IDESC_S, k > 0);
            }
            ptx::mma_commit(bar_s);
        }

        // (d) k5a mask from CB: rows t = 32*quarter + lane, columns 64*half .. +63.
        // Row quarter q = `quarter` uses the reference row r = 32q:
        //   e^{cs_t - cs_s} dt_s = u_t v_q(s),  u_t = e^{cs_t - cs_r} <= 1,  v_q(s) = e^{cs_r - cs_s} dt_s.
        // "Factored" quarters (decay across the quarter <= kMaxFactorLog) store
        // M'[t][s] = CB v_q(s) (+ D/u_t on the diagonal) and the epilogue scales the
        // row by u_t; other quarters store the exact M (u_t applied here, per entry).
        if (it == 0) wait_local(&bars[1], 0, prm.status);
        ptx::tc_fence_after();
        {
            const int t = quarter * 32 + lane;
            const float cs_t = cs[t];
            const float cs_r = cs[32 * quarter];
            const bool factored = (cs_r - cs[32 * quarter + 31]) <= kMaxFactorLog;  // warp-uniform
            const float D_h = tD[j];
            const float u_t = __expf(cs_t - cs_r);
            const float* vq = vt + quarter * kT;
            uint8_t* mblk = slot_base + K::SM + half * kTile;
            // strictly-upper tiles stay zero once written, unless sM is reused for sH
            const bool write_zeros = (K::SH == K::SM) || it == 0;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int k = 2 * half + kk;  // 32-column tile index along s
                if (k > quarter) {
                    if (write_zeros) {
                        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj)
                            *reinterpret_cast<uint4*>(mblk + ptx::swz128(t, kk * 4 + jj)) = z;
                    }
                    continue;
                }
                uint32_t r[32];
                ptx::tmem_ld32(tmem + lane_base + K::COL_CB + 32 * k, r);
                ptx::tmem_wait_ld(r);
                uint32_t pk[16];
                if (k < quarter) {
                    const float sc = factored ? 1.f : u_t;
#pragma unroll
                    for (int e4 = 0; e4 < 8; ++e4) {
                        const float4 v4 = *reinterpret_cast<const float4*>(vq + 32 * k + 4 * e4);
                        pk[2 * e4] = pack_bf16x2(__uint_as_float(r[4 * e4]) * (sc * v4.x),
                                                 __uint_as_float(r[4 * e4 + 1]) * (sc * v4.y));
                        pk[2 * e4 + 1] = pack_bf16x2(__uint_as_float(r[4 * e4 + 2]) * (sc * v4.z),
                                                     __uint_as_float(r[4 * e4 + 3]) * (sc * v4.w));
                    }
                } else if (factored) {
                    // diagonal tile, factored: causal select, D/u_t on the diagonal
                    const float d_over_u = D_h / u_t;
#pragma unroll
                    for (int e4 = 0; e4 < 8; ++e4) {
                        const float4 v4 = *reinterpret_cast<const float4*>(vq + 32 * k + 4 * e4);
                        const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
                        float m4[4];
#pragma unroll
                        for (int q2 = 0; q2 < 4; ++q2) {
                            const int c = 4 * e4 + q2;  // column inside the tile; the row is `lane`
                            const float m = __uint_as_float(r[c]) * vv[q2];
                            m4[q2] = c < lane ? m : (c == lane ? m + d_over_u : 0.f);
                        }
                        pk[2 * e4] = pack_bf16x2(m4[0], m4[1]);
                        pk[2 * e4 + 1] = pack_bf16x2(m4[2], m4[3]);
                    }
                } else {
                    // diagonal tile, exact: decay below the diagonal, D on it, zeros above
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float m2[2];
#pragma unroll
                        for (int q2 = 0; q2 < 2; ++q2) {
                            const int c = 2 * e + q2;
                            const int s = 32 * k + c;
                            const float cb = __uint_as_float(r[c]);
                            const float decay = __expf(fminf(cs_t - cs[s], 0.f));
                            const float below = cb * decay * dts[s];
                            const float diag = fmaf(cb, dts[s], D_h);
                            m2[q2] = c < lane ? below : (c == lane ? diag : 0.f);
                        }
                        pk[e] = pack_bf16x2(m2[0], m2[1]);
                    }
                }
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    *reinterpret_cast<uint4*>(mblk + ptx::swz128(t, kk * 4 + jj)) =
                        make_uint4(pk[4 * jj], pk[4 * jj + 1], pk[4 * jj + 2], pk[4 * jj + 3]);
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        ptx::named_sync(1 + slot, 256);

        // (e) k5a: Yd = M . X  (M = t, N = p, K = s; A K-major, B MN-major)
        if (leader) {
            ptx::tc_fence_after();
            const uint64_t dsc_m = ptx::desc_sw128(slot_addr + K::SM, 16, 1024);     // M, K-major
            const uint64_t dsc_x = ptx::desc_sw128(slot_addr + K::SX, kTile, 1024);  // X, MN-major
#pragma unroll
            for (int k = 0; k < kT / 16; ++k)
                ptx::mma_bf16(tmem + K::col_d(slot), dsc_m + kmaj(k), dsc_x + mnmaj(k), IDESC_D, k > 0);
            ptx::mma_commit(bar_d);
        }

        // (f) k4: s_in from the previous block (tagged words: each 64-bit word
        // holds a value and the tag of the block that wrote it, so a word with
        // the expected tag is valid by itself; no flag or fence is needed),
        // s_out = e^{cs_end} s_in + S published the same way, s_in^T to sH in bf16.
        bool my_ok = true;
        {
            const float a_blk = tEt[j * kT + kT - 1];  // e^{cs_end}
            const bool last = (blk == prm.nblk - 1);
#pragma unroll 1
            for (int mt = 0; mt < NST / 128; ++mt) {
                const int n = n0 + 128 * mt;
                float hin[32];
                if (blk == 0) {
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        const int p = half * 32 + jj;
                        hin[jj] = prm.init ? prm.init[fs_base + static_cast<size_t>(p) * NST + n] : 0.f;
                    }
                } else {
                    load_words(mt);
                    uint32_t missing = 0;
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj)
                        if (static_cast<uint32_t>(w[jj] >> 32) != want) missing |= 1u << jj;
                    if (missing) {
                        // the previous block is still writing (or failed): poll the missing
                        // words until they carry the expected tag, a poison tag, or time runs out
                        const uint64_t t_start = ptx::globaltimer_ns();
                        bool poisoned = false;
                        while (missing && !poisoned) {
                            if (ptx::globaltimer_ns() - t_start > prm.chain_wait_ns) break;
                            __nanosleep(32);
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                if (missing & (3u << (2 * i))) {
                                    ptx::ld_relaxed_2xb64(prev + (static_cast<size_t>(16 * half + i) * NST + n) * 2,
                                                          w[2 * i], w[2 * i + 1]);
#pragma unroll
                                    for (int e = 0; e < 2; ++e) {
                                        const uint32_t tg = static_cast<uint32_t>(w[2 * i + e] >> 32);
                                        if (tg == want) missing &= ~(1u << (2 * i + e));
                                        poisoned |= (tg == kPoison);
                                    }
                                }
                            }
                        }
                        if (missing) my_ok = false;
                    }
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) hin[jj] = __uint_as_float(static_cast<uint32_t>(w[jj]));
                }
                if (mt == 0) {
                    wait_local(bar_s, ph, prm.status);
                    if (K::SH == K::SM) wait_local(bar_d, ph, prm.status);  // sH shares sM with k5a's operand
                    ptx::tc_fence_after();
                }
                uint32_t r[32];
                ptx::tmem_ld32(tmem + lane_base + K::col_s(slot) + 64 * mt + half * 32, r);
                ptx::tmem_wait_ld(r);
                const uint64_t tag_hi = static_cast<uint64_t>(my_ok ? mine_tag : kPoison) << 32;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float o0 = fmaf(a_blk, hin[2 * i], __uint_as_float(r[2 * i]));
                    const float o1 = fmaf(a_blk, hin[2 * i + 1], __uint_as_float(r[2 * i + 1]));
                    ptx::st_relaxed_2xb64(mine + (static_cast<size_t>(16 * half + i) * NST + n) * 2,
                                          tag_hi | __float_as_uint(o0), tag_hi | __float_as_uint(o1));
                    if (last && prm.final_state) {
                        prm.final_state[fs_base + static_cast<size_t>(32 * half + 2 * i) * NST + n] = o0;
                        prm.final_state[fs_base + static_cast<size_t>(32 * half + 2 * i + 1) * NST + n] = o1;
                    }
                }
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    uint4 o;
                    o.x = pack_bf16x2(hin[8 * jj + 0], hin[8 * jj + 1]);
                    o.y = pack_bf16x2(hin[8 * jj + 2], hin[8 * jj + 3]);
                    o.z = pack_bf16x2(hin[8 * jj + 4], hin[8 * jj + 5]);
                    o.w = pack_bf16x2(hin[8 * jj + 6], hin[8 * jj + 7]);
                    *reinterpret_cast<uint4*>(slot_base + K::SH + ptx::swz128(n, half * 4 + jj)) = o;
                }
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        const bool chain_ok = ptx::named_sync_and(1 + slot, 256, my_ok);
        if (leader && !chain_ok) atomicOr(prm.status, 1u);

        // (g) leader: k5b Yo = C . s_in^T (M = t, N = p, K = n; A K-major, B MN-major)
        // into S's columns; refill sX for the slot's next head once k5a has read it.
        if (leader) {
            if (chain_ok) {
                ptx::tc_fence_after();
                const uint64_t dsc_c_k = ptx::desc_sw128(sbase + K::OFF_C, 16, 1024);     // C, K-major
                const uint64_t dsc_h = ptx::desc_sw128(slot_addr + K::SH, kTile, 1024);  // s_in^T, MN-major
#pragma unroll
                for (int k = 0; k < NST / 16; ++k)
                    ptx::mma_bf16(tmem + K::col_o(slot), dsc_c_k + kmaj(k), dsc_h + mnmaj(k), IDESC_O, k > 0);
                ptx::mma_commit(bar_o);
            }
            wait_local(bar_d, ph, prm.status);
            if (j + K::SLOTS < hpu) {
                ptx::mbar_arrive_expect_tx(bar_x, kTile);
                ptx::tma_load_4d(slot_base + K::SX, &tm_x, bar_x, 0, h + K::SLOTS, t0, b);
            }
        }

        // (h) epilogue: y = e^{cs_t} Yo + u_t Yd' (u_t = 1 for exact quarters), staged in sY, TMA store
        wait_local(bar_d, ph, prm.status);
        if (chain_ok) {
            wait_local(bar_o, ph, prm.status);
            ptx::tc_fence_after();
            const int t = quarter * 32 + lane;
            const float e_t = tEt[j * kT + t];
            const float cs_r = cs[32 * quarter];
            const float u_eff = (cs_r - cs[32 * quarter + 31]) <= kMaxFactorLog ? __expf(cs[t] - cs_r) : 1.f;
            uint32_t ro[32], rd[32];
            ptx::tmem_ld32(tmem + lane_base + K::col_o(slot) + half * 32, ro);
            ptx::tmem_ld32(tmem + lane_base + K::col_d(slot) + half * 32, rd);
            ptx::tmem_wait_ld(ro);
            ptx::tmem_wait_ld(rd);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c0 = 8 * jj + 2 * e;
                    pk[e] = pack_bf16x2(fmaf(e_t, __uint_as_float(ro[c0]), u_eff * __uint_as_float(rd[c0])),
                                        fmaf(e_t, __uint_as_float(ro[c0 + 1]), u_eff * __uint_as_float(rd[c0 + 1])));
                }
                *reinterpret_cast<uint4*>(slot_base + K::SY + ptx::swz128(t, half * 4 + jj)) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        ptx::named_sync(1 + slot, 256);
        if (leader && chain_ok) {
            ptx::tma_store_4d(&tm_y, slot_base + K::SY, 0, h, t0, b);
            ptx::bulk_commit_group();
        }
    }
    if (leader) ptx::bulk_wait_group_read0();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 0) ptx::tmem_dealloc(tmem, K::TMEM_COLS);
}

// ---------------------------------------------------------------- host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 4-D bf16 map over a [outer, rows, mid, inner] row-major tensor, box {64, 1, 128, 1}.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t mid, uint64_t rows, uint64_t outer) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {inner, mid, rows, outer};
    const cuuint64_t strides[3] = {inner * 2, mid * inner * 2, rows * mid * inner * 2};
    const cuuint32_t box[4] = {64, 1, kT, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t tc_counters_bytes(const ssd_dims&) { return kWorkspaceAlign; }

std::atomic<uint32_t> g_epoch{0};

// Heads per unit: the largest of 8, 4, 2, 1 that divides the heads of one group.
int heads_per_unit(const ssd_dims& d) {
    const int64_t r = d.nheads / d.ngroups;
    for (int c = kMaxHeads; c > 1; c >>= 1)
        if (r % c == 0) return c;
    return 1;
}

template <int NST>
ssd_status launch(const FwdArgs& a, void* ws) {
    using K = Cfg<NST>;
    const ssd_dims& d = a.d;
    CUtensorMap tx, tb, tc, ty;
    if (!make_map(&tx, a.x, d.headdim, d.nheads, d.seqlen, d.batch) ||
        !make_map(&tb, a.B, d.dstate, d.ngroups, d.seqlen, d.batch) ||
        !make_map(&tc, a.C, d.dstate, d.ngroups, d.seqlen, d.batch) ||
        !make_map(&ty, a.y, d.headdim, d.nheads, d.seqlen, d.batch))
        return SSD_ERR_CUDA;
    const size_t counters = tc_counters_bytes(d);
    if (cudaMemsetAsync(ws, 0, counters, a.stream) != cudaSuccess) return SSD_ERR_CUDA;
    TcParams p;
    p.dt = a.dt;
    p.dt_bias = a.dt_bias;
    p.A = a.A;
    p.D = a.D;
    p.init = a.init;
    p.final_state = a.final_state;
    p.ticket = static_cast<uint32_t*>(ws);
    p.slots = reinterpret_cast<uint64_t*>(static_cast<char*>(ws) + counters);
    p.epoch = g_epoch.fetch_add(1, std::memory_order_relaxed);
    p.status = a.status_word;
    p.batch = static_cast<int>(d.batch);
    p.H = static_cast<int>(d.nheads);
    p.G = static_cast<int>(d.ngroups);
    p.nblk = static_cast<int>((d.seqlen + kT - 1) / kT);
    p.hpu = heads_per_unit(d);
    p.ngrp = p.H / p.hpu;
    p.L = d.seqlen;
    p.chain_wait_ns = a.wait_limit_ns;
    if (cudaFuncSetAttribute(ssd_tc_fused<NST>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(K::SMEM_BYTES)) != cudaSuccess)
        return SSD_ERR_CUDA;
    const long long units = static_cast<long long>(p.nblk) * d.batch * p.ngrp;
    ssd_tc_fused<NST><<<static_cast<unsigned>(units), K::THREADS, K::SMEM_BYTES, a.stream>>>(tx, tb, tc, ty, p);
    note_launches(1);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

bool tc_supported(const ssd_dims& d, ssd_dtype io, int chunk_len) {
    if (io != SSD_BF16) return false;
    if (d.headdim != kP) return false;
    if (d.dstate != 128 && d.dstate != 256) return false;
    if (chunk_len != 128 && chunk_len != 256) return false;
    const long long nblk = (d.seqlen + kT - 1) / kT;
    if (nblk >= 65535) return false;  // state tags carry the block index in 16 bits
    if (nblk * d.batch * d.nheads >= (1ll << 31)) return false;
    if (d.seqlen >= (1ll << 31) || d.batch >= (1ll << 31) || d.nheads >= (1 << 20)) return false;
    return true;
}

size_t tc_workspace_bytes(const ssd_dims& d, int /*chunk_len*/) {
    const size_t slots = sizeof(uint64_t) * static_cast<size_t>(d.batch * d.nheads) * 2 * kP * d.dstate;
    return tc_counters_bytes(d) + align_up(slots, kWorkspaceAlign);
}

ssd_status tc_forward(const FwdArgs& a, void* ws, size_t ws_bytes) {
    if (ws_bytes < tc_workspace_bytes(a.d, a.chunk_len)) return SSD_ERR_WORKSPACE;
    for (const void* p : {a.x, static_cast<const void*>(a.B), static_cast<const void*>(a.C),
                          static_cast<const void*>(a.y)})
        if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return SSD_ERR_UNSUPPORTED;
    if (a.d.dstate == 128) return launch<128>(a, ws);
    return launch<256>(a, ws);
}

}  // namespace ssd
