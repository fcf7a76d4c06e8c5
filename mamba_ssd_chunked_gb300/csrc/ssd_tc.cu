// Fused tcgen05/TMA path of the SSD forward (bf16 io, fp32 accumulation).
//
// Work unit: one 128-token block of one batch row for a group of up to 8
// heads that read the same B/C group. Units are handed out by an atomic
// ticket in block-major order (every batch row and head group of block k
// before any unit of block k+1), so a unit only ever waits on units that
// took their tickets earlier.
//
// Per unit the CTA loads B and C once and computes C.B^T once; its heads are
// then processed by SLOTS "slots" (256 threads each) that take alternate
// heads, so one slot's waits overlap the other's work. Helper warps keep
// latency off the slots: one MMA warp issues every tcgen05.mma on the slots'
// requests, and one state agent per slot moves chunk states between global
// memory and the slot's staging buffer with bulk copies.
// Per head the five stages of the chunked SSD (burn-mamba
// "mamba2/ssd/serial.rs" k1..k5; fla "mamba2.py" naive chunked SSD) run as:
//
//   k1  dt = softplus(dt_raw + dt_bias), cs = inclusive cumsum of dt*A   (per unit, all heads)
//   k2  CB = C . B^T                 [128 x 128, K = dstate]   once per unit, tcgen05 -> TMEM
//   k3  S^T = B^T . diag(dt e^{cs_end-cs}) . X   [dstate x 64, K = 128]   tcgen05 -> TMEM
//   k5a Yd = (L o CB o dt + D I) . X [128 x 64, K = 128]       mask in registers -> TMEM, tcgen05
//   k4  s_out = e^{cs_end} s_in + S  fp32, chained through global memory (flag per block)
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
// two halves is passed like any other block boundary.
//
// Chunk-state passing: block blk of chain (b, h) reads s_in from global slot
// (chain, (blk-1) & 1) once flag (chain, (blk-1) & 1) reads blk, and publishes
// s_out to slot (chain, blk & 1), then (after its bulk store completes and a
// fence) sets that flag to blk + 1. A block only waits on an earlier ticket.
// The state agent of each slot does the polling, the bulk copies and the
// fence, so the slot's threads only touch shared memory.
//
// Operand staging (128-byte swizzle throughout; see ptx.cuh):
//   sB [t][n]  (TMA, per unit)   B operand of k2 (K-major), A operand of k3 (MN-major)
//   sC [t][n]  (TMA, per unit)   A operand of k2 and k5b (K-major)
//   per slot:
//   sX [t][p]  (TMA, per head)   B operand of k5a (MN-major, K = t)
//   sW [t][p]  (threads)         dt e^{cs_end-cs} X, B operand of k3 (MN-major)
//   sH [n][p]  (threads)         s_in in bf16, B operand of k5b (MN-major): in sW (dstate 128)
//                                or across sX and sW (dstate 256)
//   sY [t][p]  (threads)         y tile for the TMA store, in sW (after k5b has read sH)
//   sT [p][n]  (bulk copies)     fp32 state staging, one 128-column tile of the state at a time
//   TMEM: C.B^T (fp32), per slot the masked matrix M (bf16, A operand of k5a), S^T / Yo, Yd.
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
constexpr uint32_t kStateTile = kP * 128 * 4;  // fp32 state tile: 64 rows p x 128 columns n (32 KB)
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
    static constexpr int MT = NST / 128;                    // 128-row state tiles
    static constexpr int SLOTS = (NST == 128) ? 2 : 1;
    static constexpr int MATH_THREADS = 256 * SLOTS;        // the slots
    static constexpr int MMA_WARP = MATH_THREADS / 32;      // then the MMA warp, then one agent per slot
    static constexpr int THREADS = MATH_THREADS + 32 + 32 * SLOTS;
    static constexpr int NBARS = 2 + 9 * SLOTS;
    static constexpr uint32_t OFF_B = 0;
    static constexpr uint32_t OFF_C = OFF_B + NKB * kTile;
    static constexpr uint32_t OFF_SLOT = OFF_C + NKB * kTile;
    static constexpr uint32_t SLOT_BYTES = 2 * kTile + kStateTile;  // X, W, state tile
    static constexpr uint32_t SX = 0, SW = kTile, ST = 2 * kTile;   // offsets inside a slot
    static constexpr uint32_t SH = (NST == 128) ? SW : SX;          // dstate 256: sH spans sX and sW
    static constexpr uint32_t SY = SW;
    static constexpr uint32_t OFF_MISC = OFF_SLOT + SLOTS * SLOT_BYTES;
    // misc: 4 per-head tables [kMaxHeads][128] floats, per-slot v tables [4][128], scan totals
    static constexpr uint32_t TAB_BYTES = 4 * kMaxHeads * kT * 4;
    static constexpr uint32_t V_BYTES = SLOTS * 4 * kT * 4;
    static constexpr uint32_t MISC_BYTES = TAB_BYTES + V_BYTES + 512 + 512;
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + MISC_BYTES + 1024;  // + alignment slack
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_CB = 0;
    // per slot: M (64 packed bf16 columns), S^T (64 per state tile; Yo reuses it), Yd (64)
    __host__ __device__ static constexpr uint32_t col_m(int slot) { return 128 + (128 + 64 * MT) * slot; }
    __host__ __device__ static constexpr uint32_t col_s(int slot) { return col_m(slot) + 64; }
    __host__ __device__ static constexpr uint32_t col_d(int slot) { return col_s(slot) + 64 * MT; }
    __host__ __device__ static constexpr uint32_t col_o(int slot) { return col_s(slot); }
    static_assert(col_d(SLOTS - 1) + 64 <= TMEM_COLS, "tensor memory budget");
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
    float* slots;          // [batch*H][2][MT][P][128] fp32 chained states
    uint32_t* flags;       // [batch*H][2]: block index + 1 of the state in the slot (kPoison: failed)
    uint32_t* ticket;      // block-major work counter
    uint32_t* status;      // device status word
    int batch, H, G, nblk, hpu, ngrp;  // hpu heads per unit, ngrp = H / hpu head groups
    long long L;
    unsigned long long chain_wait_ns;  // limit on waiting for the previous block's state
    float dt_min, dt_max;              // clamp of softplus(dt + dt_bias)
    const int32_t* seq;                // [batch, L] packed-sequence ids, or null
};

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
    // bars: [0] B/C landed, [1] CB done; per slot s at 2 + 9s: X landed, S done, Yd done, Yo done,
    // requests to the MMA warp (W ready: k3, M ready: k5a, s_in ready: k5b), state tile landed
    // (agent -> slot), state tile staged (slot -> agent)
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(bars + K::NBARS);
    int* sInfo = reinterpret_cast<int*>(sTmem + 1);  // [0] unit, [1+s] skip k5b, [3+s] chain failed

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool is_math = tid < K::MATH_THREADS;
    const int slot = is_math ? (tid >> 8) : 0, stid = tid & 255, swarp = stid >> 5;
    const int quarter = warp & 3, half = swarp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;

    if (tid == 0) {
        sInfo[0] = static_cast<int>(atomicAdd(prm.ticket, 1u));
#pragma unroll
        for (int i = 0; i < K::NBARS; ++i) ptx::mbar_init(&bars[i], 1);
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
    const bool last_blk = (blk == prm.nblk - 1);
    const uint32_t sbase = ptx::smem_u32(smem);
    uint8_t* slot_base = smem + K::OFF_SLOT + slot * K::SLOT_BYTES;
    auto bar_of = [&](int sl, int k) { return &bars[2 + 9 * sl + k]; };
    uint64_t* bar_x = bar_of(slot, 0);
    uint64_t* bar_s = bar_of(slot, 1);
    uint64_t* bar_d = bar_of(slot, 2);
    uint64_t* bar_o = bar_of(slot, 3);
    uint64_t* req_s = bar_of(slot, 4);
    uint64_t* req_d = bar_of(slot, 5);
    uint64_t* req_o = bar_of(slot, 6);
    uint64_t* bar_st = bar_of(slot, 7);
    uint64_t* bar_pub = bar_of(slot, 8);
    const bool leader = is_math && stid == 0;
    // the unit is a real (block, batch row, head group) and its heads share one B/C group
    SSD_CHECK(prm.status, b < prm.batch && blk < prm.nblk && h0 + hpu <= prm.H && hpu <= kMaxHeads && g < prm.G &&
                              (h0 + hpu - 1) / (prm.H / prm.G) == g && slot < K::SLOTS);

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
        if (t < L)
            dtv = fminf(fmaxf(softplus_f(prm.dt[(static_cast<long long>(b) * L + t) * prm.H + h] + prm.dt_bias[h]),
                              prm.dt_min),
                        prm.dt_max);
        float v = dtv * prm.A[h];
        // a new packed sequence starts at t: no state crosses (kSeqCutNats)
        if (prm.seq && t > 0 && t < L && prm.seq[static_cast<long long>(b) * L + t] != prm.seq[static_cast<long long>(b) * L + t - 1])
            v -= kSeqCutNats;
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

    constexpr uint32_t IDESC_CB = ptx::idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t IDESC_S = ptx::idesc_bf16_f32(128, 64, true, true);
    constexpr uint32_t IDESC_D = ptx::idesc_bf16_f32(128, 64, false, true);
    constexpr uint32_t IDESC_O = ptx::idesc_bf16_f32(128, 64, false, true);
    // Matrix descriptors are built once per issue from the operand base; a K
    // step adds its byte offset to the start-address field (offsets stay far
    // below the field's range).
    auto kmaj = [](int k) { return static_cast<uint64_t>(((k >> 2) * kTile + (k & 3) * 32) >> 4); };
    auto mnmaj = [](int k) { return static_cast<uint64_t>((k * 2048) >> 4); };
    auto heads_of = [&](int sl) { return sl < hpu ? (hpu - sl + K::SLOTS - 1) / K::SLOTS : 0; };

    if (warp == K::MMA_WARP) {
        // ---- the MMA warp: k2 once, then k3 / k5a / k5b for each head on the slots' requests
        if (lane == 0) {
            wait_local(&bars[0], 0, prm.status);
            ptx::tc_fence_after();
            const uint64_t dsc_c_k = ptx::desc_sw128(sbase + K::OFF_C, 16, 1024);     // C, K-major
            const uint64_t dsc_b_k = ptx::desc_sw128(sbase + K::OFF_B, 16, 1024);     // B, K-major
            const uint64_t dsc_b_mn = ptx::desc_sw128(sbase + K::OFF_B, kTile, 1024);  // B^T, MN-major
#pragma unroll
            for (int k = 0; k < NST / 16; ++k)
                ptx::mma_bf16(tmem + K::COL_CB, dsc_c_k + kmaj(k), dsc_b_k + kmaj(k), IDESC_CB, k > 0);
            ptx::mma_commit(&bars[1]);
            // Requests arrive per slot in the order k3, k5a, k5b for each of the slot's heads.
            int nh[K::SLOTS], done[K::SLOTS], stage[K::SLOTS];
            int pending = 0;
#pragma unroll
            for (int sl = 0; sl < K::SLOTS; ++sl) {
                nh[sl] = heads_of(sl);
                done[sl] = 0;
                stage[sl] = 0;
                pending += 3 * nh[sl];
            }
            uint64_t idle_since = ptx::globaltimer_ns();
            while (pending > 0) {
                bool progressed = false;
#pragma unroll
                for (int sl = 0; sl < K::SLOTS; ++sl) {
                    if (done[sl] >= nh[sl]) continue;
                    if (!ptx::mbar_test_wait(bar_of(sl, 4 + stage[sl]), done[sl] & 1)) continue;
                    ptx::tc_fence_after();
                    const uint32_t saddr = sbase + K::OFF_SLOT + sl * K::SLOT_BYTES;
                    if (stage[sl] == 0) {
                        // k3: S^T = B^T . W  (M = n, N = p, K = t; both MN-major)
                        const uint64_t dsc_w = ptx::desc_sw128(saddr + K::SW, kTile, 1024);
#pragma unroll
                        for (int mt = 0; mt < K::MT; ++mt)
#pragma unroll
                            for (int k = 0; k < kT / 16; ++k)
                                ptx::mma_bf16(tmem + K::col_s(sl) + 64 * mt,
                                              dsc_b_mn + ((2 * mt * kTile) >> 4) + mnmaj(k), dsc_w + mnmaj(k),
                                              IDESC_S, k > 0);
                        ptx::mma_commit(bar_of(sl, 1));
                    } else if (stage[sl] == 1) {
                        // k5a: Yd = M . X  (M = t, N = p, K = s; A from TMEM, B MN-major)
                        const uint64_t dsc_x = ptx::desc_sw128(saddr + K::SX, kTile, 1024);
#pragma unroll
                        for (int k = 0; k < kT / 16; ++k)
                            ptx::mma_bf16_ta(tmem + K::col_d(sl), tmem + K::col_m(sl) + 8 * k, dsc_x + mnmaj(k),
                                             IDESC_D, k > 0);
                        ptx::mma_commit(bar_of(sl, 2));
                    } else {
                        // k5b: Yo = C . s_in^T  (M = t, N = p, K = n; A K-major, B MN-major), into S's columns
                        if (!sInfo[1 + sl]) {
                            const uint64_t dsc_h = ptx::desc_sw128(saddr + K::SH, kTile, 1024);
#pragma unroll
                            for (int k = 0; k < NST / 16; ++k)
                                ptx::mma_bf16(tmem + K::col_o(sl), dsc_c_k + kmaj(k), dsc_h + mnmaj(k), IDESC_O,
                                              k > 0);
                        }
                        ptx::mma_commit(bar_of(sl, 3));
                    }
                    if (++stage[sl] == 3) {
                        stage[sl] = 0;
                        ++done[sl];
                    }
                    --pending;
                    progressed = true;
                }
                const uint64_t now = ptx::globaltimer_ns();
                if (progressed) {
                    idle_since = now;
                } else if (now - idle_since > 2 * kLocalWaitNs) {
                    atomicOr(prm.status, 2u);  // a slot stopped requesting: give up
                    break;
                }
            }
        }
        __syncwarp();
    } else if (!is_math) {
        // ---- state agent of slot `sl`: fetch s_in tiles, publish s_out tiles and the block's flag
        const int sl = warp - K::MMA_WARP - 1;
        if (lane == 0) {
            uint8_t* st_buf = smem + K::OFF_SLOT + sl * K::SLOT_BYTES + K::ST;
            uint64_t* a_st = bar_of(sl, 7);
            uint64_t* a_pub = bar_of(sl, 8);
            uint32_t ph_pub = 0;
            const int nh = heads_of(sl);
            for (int q = 0; q < nh; ++q) {
                const int h = h0 + sl + q * K::SLOTS;
                const int chain = b * prm.H + h;
                SSD_CHECK(prm.status, h < h0 + hpu && chain < prm.batch * prm.H && sl < K::SLOTS);
                bool fail = false;
                if (blk > 0) {
                    const uint32_t* pf = prm.flags + chain * 2 + ((blk - 1) & 1);
                    const uint32_t want = static_cast<uint32_t>(blk);
                    uint32_t v = ptx::ld_relaxed_gpu(pf);
                    if (v != want) {
                        const uint64_t t_start = ptx::globaltimer_ns();
                        while (v != want && v != kPoison) {
                            if (ptx::globaltimer_ns() - t_start > prm.chain_wait_ns) break;
                            __nanosleep(64);
                            v = ptx::ld_relaxed_gpu(pf);
                        }
                    }
                    fail = (v != want);
                    if (!fail) {
                        ptx::fence_acquire_gpu();
                        ptx::fence_proxy_async_global();  // the bulk loads below read what the flag guards
                    }
                }
                sInfo[3 + sl] = fail ? 1 : 0;
                const float* prev =
                    prm.slots + (static_cast<size_t>(chain) * 2 + ((blk - 1) & 1)) * K::MT * (kStateTile / 4);
                float* mine = prm.slots + (static_cast<size_t>(chain) * 2 + (blk & 1)) * K::MT * (kStateTile / 4);
                const size_t fs_base = static_cast<size_t>(chain) * kP * NST;
#pragma unroll 1
                for (int mt = 0; mt < K::MT; ++mt) {
                    // fetch s_in tile mt into the staging buffer
                    if (fail || (blk == 0 && !prm.init)) {
                        ptx::mbar_arrive(a_st);  // nothing to load: the slot uses zeros (or gives up)
                    } else if (blk == 0) {
                        ptx::mbar_arrive_expect_tx(a_st, kStateTile);
                        if (K::MT == 1) {
                            ptx::bulk_load(st_buf, prm.init + fs_base, kStateTile, a_st);
                        } else {
                            for (int p = 0; p < kP; ++p)
                                ptx::bulk_load(st_buf + p * 512,
                                               prm.init + fs_base + static_cast<size_t>(p) * NST + 128 * mt, 512, a_st);
                        }
                    } else {
                        ptx::mbar_arrive_expect_tx(a_st, kStateTile);
                        ptx::bulk_load(st_buf, prev + static_cast<size_t>(mt) * (kStateTile / 4), kStateTile, a_st);
                    }
                    // the slot stages s_out tile mt in place; write it out
                    wait_local(a_pub, ph_pub, prm.status);
                    ph_pub ^= 1;
                    if (!fail) {
                        if (!last_blk) {
                            ptx::bulk_store(mine + static_cast<size_t>(mt) * (kStateTile / 4), st_buf, kStateTile);
                        } else if (prm.final_state) {
                            if (K::MT == 1) {
                                ptx::bulk_store(prm.final_state + fs_base, st_buf, kStateTile);
                            } else {
                                for (int p = 0; p < kP; ++p)
                                    ptx::bulk_store(prm.final_state + fs_base + static_cast<size_t>(p) * NST + 128 * mt,
                                                    st_buf + p * 512, 512);
                            }
                        }
                        ptx::bulk_commit_group();
                        ptx::bulk_wait_group_read0();  // the staging buffer may be refilled
                    }
                }
                // the state is in global memory before the flag says so
                ptx::bulk_wait_group0();
                if (!last_blk) {
                    ptx::fence_proxy_async_global();
                    __threadfence();
                    ptx::st_relaxed_gpu(prm.flags + chain * 2 + (blk & 1),
                                        fail ? kPoison : static_cast<uint32_t>(blk + 1));
                }
                if (fail) atomicOr(prm.status, 1u);
            }
        }
        __syncwarp();
    }

    // ---- per-slot head loop
    bool b_ready = false;  // this thread has seen B/C land
    int it = 0;
    for (int j = slot; is_math && j < hpu; j += K::SLOTS, ++it) {
        const int h = h0 + j;
        const uint32_t ph = it & 1;
        const float* cs = tCs + j * kT;
        const float* dts = tDt + j * kT;
        const float* wts = tWt + j * kT;
        float* vt = tV + slot * 4 * kT;
        float* st_buf = reinterpret_cast<float*>(slot_base + K::ST);

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

        // (c) k3 is issued by the MMA warp
        if (leader) ptx::mbar_arrive(req_s);

        // (d) k5a mask from CB: rows t = 32*quarter + lane, columns 64*half .. +63, into TMEM.
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
            uint32_t pk[32];  // this thread's 64 columns of M as packed bf16 pairs
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int k = 2 * half + kk;  // 32-column tile index along s
                if (k > quarter) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) pk[16 * kk + e] = 0u;
                    continue;
                }
                uint32_t r[32];
                ptx::tmem_ld32(tmem + lane_base + K::COL_CB + 32 * k, r);
                ptx::tmem_wait_ld(r);
                if (k < quarter) {
                    const float sc = factored ? 1.f : u_t;
#pragma unroll
                    for (int e4 = 0; e4 < 8; ++e4) {
                        const float4 v4 = *reinterpret_cast<const float4*>(vq + 32 * k + 4 * e4);
                        pk[16 * kk + 2 * e4] = pack_bf16x2(__uint_as_float(r[4 * e4]) * (sc * v4.x),
                                                           __uint_as_float(r[4 * e4 + 1]) * (sc * v4.y));
                        pk[16 * kk + 2 * e4 + 1] = pack_bf16x2(__uint_as_float(r[4 * e4 + 2]) * (sc * v4.z),
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
                        pk[16 * kk + 2 * e4] = pack_bf16x2(m4[0], m4[1]);
                        pk[16 * kk + 2 * e4 + 1] = pack_bf16x2(m4[2], m4[3]);
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
                        pk[16 * kk + e] = pack_bf16x2(m2[0], m2[1]);
                    }
                }
            }
            ptx::tmem_st32(tmem + lane_base + K::col_m(slot) + 32 * half, pk);
            ptx::tmem_wait_st();
        }
        ptx::tc_fence_before();
        ptx::named_sync(1 + slot, 256);

        // (e) k5a is issued by the MMA warp
        if (leader) ptx::mbar_arrive(req_d);

        // (f) k4: s_out = e^{cs_end} s_in + S per 128-column state tile, staged in place
        // for the agent; s_in^T to sH in bf16 for k5b. Thread (quarter, half) owns
        // state column n = 32*quarter + lane of the tile and rows p = 32*half .. +31.
        bool chain_ok = true;
        {
            const float a_blk = tEt[j * kT + kT - 1];  // e^{cs_end}
            const int nl = quarter * 32 + lane;
#pragma unroll 1
            for (int mt = 0; mt < K::MT; ++mt) {
                const uint32_t pst = static_cast<uint32_t>(it * K::MT + mt) & 1;
                wait_local(bar_st, pst, prm.status);
                chain_ok = (sInfo[3 + slot] == 0);
                const bool zero_in = !chain_ok || (blk == 0 && !prm.init);
                if (mt == 0) {
                    wait_local(bar_s, ph, prm.status);
                    if (K::SH != K::SW) wait_local(bar_d, ph, prm.status);  // sH overlays k5a's sX
                }
                ptx::tc_fence_after();
                uint32_t r[32];
                ptx::tmem_ld32(tmem + lane_base + K::col_s(slot) + 64 * mt + half * 32, r);
                ptx::tmem_wait_ld(r);
                float hin[32];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    float* cell = st_buf + (32 * half + jj) * 128 + nl;
                    hin[jj] = zero_in ? 0.f : *cell;
                    *cell = fmaf(a_blk, hin[jj], __uint_as_float(r[jj]));
                }
                const int n = nl + 128 * mt;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    uint4 o;
                    o.x = pack_bf16x2(hin[8 * jj + 0], hin[8 * jj + 1]);
                    o.y = pack_bf16x2(hin[8 * jj + 2], hin[8 * jj + 3]);
                    o.z = pack_bf16x2(hin[8 * jj + 4], hin[8 * jj + 5]);
                    o.w = pack_bf16x2(hin[8 * jj + 6], hin[8 * jj + 7]);
                    *reinterpret_cast<uint4*>(slot_base + K::SH + ptx::swz128(n, half * 4 + jj)) = o;
                }
                ptx::fence_proxy_async_smem();  // the agent's bulk store and k5b read what was written
                ptx::tc_fence_before();
                ptx::named_sync(1 + slot, 256);
                if (leader) ptx::mbar_arrive(bar_pub);
            }
        }

        // (g) k5b is issued by the MMA warp (skipped when the chain failed);
        // refill sX for the slot's next head once k5a has read it
        if (leader) {
            sInfo[1 + slot] = chain_ok ? 0 : 1;
            ptx::mbar_arrive(req_o);
            if (K::SH == K::SW) {
                wait_local(bar_d, ph, prm.status);
                if (j + K::SLOTS < hpu) {
                    ptx::mbar_arrive_expect_tx(bar_x, kTile);
                    ptx::tma_load_4d(slot_base + K::SX, &tm_x, bar_x, 0, h + K::SLOTS, t0, b);
                }
            }
        }

        // (h) epilogue: y = e^{cs_t} Yo + u_t Yd' (u_t = 1 for exact quarters), staged in sY, TMA store
        wait_local(bar_d, ph, prm.status);
        wait_local(bar_o, ph, prm.status);  // also when k5b was skipped: sH is free once this completes
        if (leader && K::SH != K::SW && j + K::SLOTS < hpu) {
            ptx::mbar_arrive_expect_tx(bar_x, kTile);
            ptx::tma_load_4d(slot_base + K::SX, &tm_x, bar_x, 0, h + K::SLOTS, t0, b);
        }
        if (chain_ok) {
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
        if (leader && chain_ok && SSD_CHECK(prm.status, h < prm.H && h >= h0 && h < h0 + hpu)) {
            ptx::tma_store_4d(&tm_y, slot_base + K::SY, 0, h, t0, b);
            ptx::bulk_commit_group();
        }
    }
    if (leader) ptx::bulk_wait_group_read0();
    ptx::tc_fence_before();
    __syncthreads();  // every slot is done, the MMA warp has committed its last group, the agents are idle
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

// Work ticket, then one flag per (chain, parity); cleared before every launch.
size_t tc_counters_bytes(const ssd_dims& d) {
    return align_up(sizeof(uint32_t) * static_cast<size_t>(1 + 2 * d.batch * d.nheads), kWorkspaceAlign);
}

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
    if (!make_map_bf16(&tx, a.x, d.headdim, d.nheads, d.seqlen, d.batch) ||
        !make_map_bf16(&tb, a.B, d.dstate, d.ngroups, d.seqlen, d.batch) ||
        !make_map_bf16(&tc, a.C, d.dstate, d.ngroups, d.seqlen, d.batch) ||
        !make_map_bf16(&ty, a.y, d.headdim, d.nheads, d.seqlen, d.batch))
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
    p.flags = p.ticket + 1;
    p.slots = reinterpret_cast<float*>(static_cast<char*>(ws) + counters);
    p.status = a.status_word;
    p.batch = static_cast<int>(d.batch);
    p.H = static_cast<int>(d.nheads);
    p.G = static_cast<int>(d.ngroups);
    p.nblk = static_cast<int>((d.seqlen + kT - 1) / kT);
    p.hpu = heads_per_unit(d);
    p.ngrp = p.H / p.hpu;
    p.L = d.seqlen;
    p.chain_wait_ns = a.wait_limit_ns;
    p.dt_min = a.dt_min;
    p.dt_max = a.dt_max;
    p.seq = a.seq_idx;
    if (cudaFuncSetAttribute(ssd_tc_fused<NST>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(K::SMEM_BYTES)) != cudaSuccess)
        return SSD_ERR_CUDA;
    const long long units = static_cast<long long>(p.nblk) * d.batch * p.ngrp;
    timing_begin(a.stream);
    ssd_tc_fused<NST><<<static_cast<unsigned>(units), K::THREADS, K::SMEM_BYTES, a.stream>>>(tx, tb, tc, ty, p);
    timing_end(a.stream);
    note_launches(1);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

bool make_map_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t mid, uint64_t rows, uint64_t outer,
                   uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {inner, mid, rows, outer};
    const cuuint64_t strides[3] = {inner * 2, mid * inner * 2, rows * mid * inner * 2};
    const cuuint32_t box[4] = {64, 1, box_rows, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_supported(const ssd_dims& d, ssd_dtype io, int chunk_len) {
    if (io != SSD_BF16) return false;
    if (d.headdim != kP) return false;
    if (d.dstate != 128 && d.dstate != 256) return false;
    if (chunk_len != 128 && chunk_len != 256) return false;
    const long long nblk = (d.seqlen + kT - 1) / kT;
    if (nblk * d.batch * d.nheads >= (1ll << 31)) return false;
    if (d.seqlen >= (1ll << 31) || d.batch >= (1ll << 31) || d.nheads >= (1 << 20)) return false;
    return true;
}

size_t tc_workspace_bytes(const ssd_dims& d, int /*chunk_len*/) {
    const size_t slots = sizeof(float) * static_cast<size_t>(d.batch * d.nheads) * 2 * kP * d.dstate;
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
