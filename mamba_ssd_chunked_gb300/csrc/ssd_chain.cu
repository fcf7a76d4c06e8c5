// Chain-local fused forward, head-pair-major form (tcgen05/TMA, bf16 io,
// dstate 128 or 256, headdim 64).
//
// A persistent CTA per SM walks a contiguous range of the flattened
// (chain, block) index space. A chain is a pair of heads of one batch row that
// read the same B/C group (paired by decay rate, chain_tables); a block is 128
// tokens. Along a chain the blocks are processed in order by the same CTA, so
// the chunk state stays in tensor memory from block to block; only where a
// CTA's range starts or ends inside a chain does a state cross to the
// neighbouring CTA: through global memory behind a flag (the hand-off), or the
// later CTA recomputes it from a zero state over the blocks in which it decays
// by kWarmupNats (the warm-up, warmup_blocks). A CTA processes the tail of its
// range (a chain start) first and the head of its range (the continuation) last.
//
// Per block the chunked SSD (burn-mamba "mamba2/ssd/serial.rs" k1..k5; fla
// "mamba2.py" naive chunked SSD) is computed with every MMA's M dimension
// running over (head, p) of the pair, 128 rows:
//
//   dt_t = clamp(softplus(dt_raw + dt_bias)), cs_t = cumsum of dt*A over the sub-block,
//   c    = cs_end / 2 (a reference log-decay per sub-block and head),
//   W_s  = X_s dt_s e^{c - cs_s}                  (bf16, built in place over X)
//   Z    = e^{c} s_in                              (fp32 state in TMEM, rows (h, p), columns n)
//   k3   Z += W^T B            ->  Z = e^{c - cs_end} s_out
//   k5a  Y^T  = W^T L^T        with L = C.B^T masked to s <= t (shared by the heads)
//   k5b  Y^T += H C^T          with H = bf16(e^{c} s_in), read by the MMA from TMEM
//   y_t  = e^{cs_t - c} Y_t + (D / wf_t) W_t     (= ... + D x_t, wf_t = dt_t e^{c - cs_t})
//
// since e^{cs_t - cs_s} dt_s X_s = e^{cs_t - c} (e^{c - cs_s} dt_s X_s) and
// e^{cs_t} C_t s_in = e^{cs_t - c} C_t (e^{c} s_in). Every factor stays within
// e^{+-d/2} for a sub-block decay d, so a block whose decay exceeds
// kMaxSubDecay is split into 2, 4 or 8 sub-blocks (64, 32 or 16 tokens) that
// each pass the state on like a block. A 16-token sub-block that still decays
// faster ("extreme") keeps the state path (with its reference moved to
// cs_end + kExtremeRef) and C s_in with reference 0, and the epilogue adds its
// intra-block sum with per-entry decays on the CUDA cores. Tokens whose W factor is
// so small that x wf may underflow bf16 take D x_t from x in global memory.
//
// L for every (batch, block, group) is computed once by a small kernel
// (chain_masks) into the workspace, and so is every job's table record (dt,
// sub-block split, per-token factors; chain_tables) with its estimated cost;
// the chain kernel streams both like inputs. Each chain CTA takes the
// contiguous job range that carries its share of the total cost (cta_range; a
// job costs more the more sub-blocks it has), so that CTAs holding
// fast-decaying heads finish with the rest. The three kernels are launched
// with programmatic stream serialization.
//
// Roles (16 warps):
//   warp 0       TMA producer: the L / B / C ring (Lay<NS>)
//   warp 1       MMA issuer, state path: k3 (at dstate 256 also the B loads)
//   warp 2       MMA issuer, output path: k5a, k5b
//   warp 3       TMA producer: X (three or two job slots of two heads) and each
//                job's table record; L2 prefetch of chain-start states and (two
//                slots) of the X a slot round ahead
//   warps 4..7   W from X in place
//   warps 8..11  state: rescale Z, write H; load / store states at segment ends
//   warps 12..15 epilogue: y from Y (TMEM) and W (shared memory), written over W
//                and stored from there by TMA
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>

#include "ptx.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kT = 128;                 // tokens per block
constexpr int kP = 64;                  // rows per chain half: a head at headdim 64, half a head at 128
constexpr int kHG = 2;                  // heads per chain
constexpr uint32_t kTile = 16384;       // 128 rows x 128 bytes, 128-byte swizzle
constexpr float kMaxSubDecay = 150.f;   // a sub-block decaying at most this keeps factors within e^{+-75}
constexpr float kExtremeRef = 75.f;     // extreme sub-blocks: state reference cs_end + this
constexpr unsigned long long kLocalWaitNs = 2000000000ull;
constexpr int kTabSlots = 4;            // table ring depth (jobs)
constexpr int kNumTab = 3;              // per-token tables per (job, head) staged in shared memory
enum Tab { TAB_WF = 0, TAB_U = 1, TAB_UG = 2 };  // W factor wf, epilogue factors u and D / wf
// Tokens with wf below this take D x from x itself: above it (D / wf) W is off from
// D x by at most |D| 5e-4 even where x wf is a bf16 subnormal (spacing 2^-133).
constexpr float kTinyWF = 1e-37f;
constexpr int kNumTabX = 2;             // per-token tables per (job, head) read from global only
enum TabX { TABX_CS = 0, TABX_DT = 1 }; // sub-block cumsum and dt (extreme sub-blocks)
constexpr int kScal = 32;               // scalars per (job, head): ec[8], hs[8], is[8], D
enum Scal { SC_EC = 0, SC_HS = 8, SC_IS = 16, SC_D = 24 };
// A continuation segment may start from a zero state this many nats of decay
// (both heads) before its first block instead of waiting for the previous CTA's
// hand-off: what the zero start leaves out is scaled by e^{-32} < 2^-46, some
// 2^-22 of one fp32 unit in the last place of the state it is added to.
constexpr float kWarmupNats = 32.f;
// A warm-up block's time as a share of its job cost, in percent (the warm-up
// decision; on the 130M and 2.7B layer shapes 60 to 70 balance best).
constexpr uint32_t kWarmupCostPct = 70;
// Decay-sorted head pairs: the pair table is sorted when nheads and the
// per-group sort stay this small (every table CTA sorts its own copy).
constexpr int kSortMaxHeads = 1024;
constexpr long long kSortMaxWork = 65536;  // nheads x heads per group
constexpr int kThreads = 512;
constexpr int kRingMax = 4;             // slots of the L / B / C ring, at most (Lay::kRing)
constexpr int kXWMax = 3;               // X / W / y job slots, at most (Lay::kXW)
// Per-job table record in the workspace: [2 heads][kNumTab][128] floats,
// [2 heads][kScal] floats, {nq, extreme, 0, 0} (the part a shared-memory slot
// holds), then [2 heads][kNumTabX][128] floats.
constexpr uint32_t kRecTab = kHG * kNumTab * kT * 4;
constexpr uint32_t kRecScal = kHG * kScal * 4;
constexpr uint32_t kRecSmem = kRecTab + kRecScal + 16;
constexpr uint32_t kRecBytes = kRecSmem + kHG * kNumTabX * kT * 4;
static_assert(kRecSmem % 16 == 0 && kRecBytes % 16 == 0, "bulk copies move multiples of 16 bytes");

// Per-dstate layout (NS = 128 or 256).
// At 128 the ring carries, per job, B, L and C, one 32 KB slot each, at
// positions kKinds J + kind in the order B, L, C: the producer issues a job's
// B as soon as k3 of the job before has freed its slot, ahead of L and C,
// whose slots k5a and k5b free later; B is what the state path (k3) waits for.
// At 256, B (both 128-column halves of n, 64 KB) has a buffer of its own,
// which the k3 issuer refills with the next job's B as soon as k3 of the job
// has read it; k3 then runs at N = 256 over the contiguous halves. The ring
// carries L and the two C halves in two slots: an entry reuses the slot of
// the entry two positions earlier, so a job's second C half waits for its own
// L, which k5a frees (k5a waits for nothing of that C half).
// TMEM (512 columns): the fp32 state Z (NS columns), kHBuf bf16 copies H of
// the scaled state (NS / 2 columns each, the A operand of k5b) and kYBuf
// output accumulators Y (128 columns each). At NS = 256 the state takes half
// of TMEM, so H and Y are single-buffered.
template <int NS>
struct Lay {
    static_assert(NS == 128 || NS == 256, "dstate 128 or 256");
    static constexpr int kNB = NS / 128;
    static constexpr bool kOwnB = NS == 256;  // B in a buffer of its own, loaded by the k3 issuer
    static constexpr int kKinds = kOwnB ? 1 + kNB : 1 + 2 * kNB;
    static constexpr int kHBuf = NS == 128 ? 2 : 1;
    static constexpr int kYBuf = NS == 128 ? 2 : 1;
    // Shared memory: kRing ring slots, the B buffer (kOwnB) and kXW X/W/y job
    // slots, six 32 KB slots in all; three jobs in flight at 128, two at 256.
    static constexpr int kRing = NS == 128 ? 3 : 2;
    static constexpr int kXW = NS == 128 ? 3 : 2;
    // L2 prefetch of the X a slot round ahead (from the second round on: the first
    // round's copies already crowd the start). It pays with two X/W slots; with three,
    // the slot frees late enough for the load itself and the prefetch only adds traffic.
    static constexpr bool kPrefetchX = kXW == 2;
    static_assert(kRing <= kRingMax && kXW <= kXWMax && kRing + (kOwnB ? kNB : 0) + kXW == 6, "six 32 KB slots");
    static constexpr uint32_t OFF_B = 2 * kRing * kTile;  // kOwnB: B as 2 kNB tiles of 64 columns of n
    static constexpr uint32_t OFF_XW = OFF_B + (kOwnB ? 2 * kNB * kTile : 0);
    static constexpr uint32_t COL_Z = 0;
    static constexpr uint32_t COL_H = NS;
    static constexpr uint32_t COL_Y = NS + kHBuf * (NS / 2);
    static_assert(COL_Y + kYBuf * 128 == 512, "TMEM budget");
    __host__ __device__ static constexpr int kindB(int half) { return kOwnB ? -1 : half; }  // ring kinds at 128 only
    __host__ __device__ static constexpr int kindL() { return kOwnB ? 0 : kNB; }
    __host__ __device__ static constexpr int kindC(int half) { return kOwnB ? 1 + half : 1 + kNB + half; }
};

struct Cfg {
    // ring of kRing 32 KB slots ([t][128] as two 64-column tiles) holding, in
    // consumption order, L and the B and C halves of each job (Lay<NS>)
    static constexpr uint32_t OFF_RING = 0;               // then the X/W slots at Lay::OFF_XW
    static constexpr uint32_t OFF_TAB = 12 * kTile;      // [slots] table records
    static constexpr uint32_t OFF_BAR = (OFF_TAB + kTabSlots * kRecSmem + 7) & ~7u;
    static constexpr int NBAR = 44;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr uint32_t OFF_SCAN = OFF_MISC + 64;  // [kThreads / 32] u64, cta_range
    static constexpr uint32_t OFF_ORDER = OFF_SCAN + 128;  // [kSortMaxHeads] the pair order (job_pos)
    static constexpr uint32_t SMEM_BYTES = OFF_ORDER + kSortMaxHeads * 4 + 1024;
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

enum Bar {
    B_R_FULL0 = 0, B_R_EMPTY0 = B_R_FULL0 + kRingMax,
    B_X_FULL0 = B_R_EMPTY0 + kRingMax, B_XW_FREE0 = B_X_FULL0 + kXWMax, B_XW_EMPTY0 = B_XW_FREE0 + kXWMax,
    B_TAB_FULL0 = B_XW_EMPTY0 + kXWMax, B_TAB_FULL3 = B_TAB_FULL0 + 3, B_TAB_EMPTY0, B_TAB_EMPTY3 = B_TAB_EMPTY0 + 3,
    B_W_FULL0, B_SCALED = B_W_FULL0 + kXWMax, B_S_DONE, B_H_FULL0, B_H_FULL1, B_H_EMPTY0, B_H_EMPTY1,
    B_Y_FULL0, B_Y_FULL1, B_Y_EMPTY0, B_Y_EMPTY1,
    B_DRAIN_K3, B_DRAIN_Y, B_B_FULL, B_B_EMPTY,
    B_COUNT
};
static_assert(B_COUNT <= Cfg::NBAR, "barrier budget");
static_assert(B_TAB_FULL3 - B_TAB_FULL0 + 1 == kTabSlots && B_TAB_EMPTY3 - B_TAB_EMPTY0 + 1 == kTabSlots,
              "one full and one empty barrier per table slot");
static_assert((kTabSlots & (kTabSlots - 1)) == 0, "table slots are indexed by J & (kTabSlots - 1)");

struct ChainParams {
    const float* dt;
    const float* dt_bias;
    const float* A;
    const float* D;
    const float* init;
    float* final_state;
    const __nv_bfloat16* x;
    __nv_bfloat16* y;
    const __nv_bfloat16* masks;  // [b][nblk][G][t][s] bf16 L tiles (read again by the extreme path)
    const uint8_t* tables;       // [chain * nblk + block] table records
    const uint8_t* cost;         // [jobs] estimated job costs (cta_range); null: even split by count
    const uint8_t* job_cost;     // [jobs] the same costs, always set (warm-up decision)
    const float2* decay;         // [jobs] (head 0, head 1) decay of the whole block, in nats
    const int* order;            // [H] heads in pair order: chain cb of a row is heads order[2 cb], order[2 cb + 1]
    int warmup;                  // 0: never warm up, 1: when the hand-off would come late, 2: whenever possible
    float* handoff;              // [nCTA][2][P][N] fp32 states handed from CTA i to CTA i + 1
    uint32_t* ticket;            // CTA order counter
    uint32_t* flags;             // [nCTA]: 1 once CTA i's hand-off state is in place
    uint32_t* status;
    int batch, H, G, nblk, nchains, ncta;
    long long L, total;          // total = nchains * nblk jobs
    unsigned long long chain_wait_ns;
    float dt_min, dt_max;        // clamp of softplus(dt + dt_bias)
};

// A job is one block of one chain. The CTA's jobs, in processing order (all
// indices fit 31 bits: the host only launches when chains * blocks < 2^31).
// The segment of chain cF (the head of the range, processed last) starts at
// block a; with wu > 0 it is preceded by wu warm-up blocks that only advance
// the state (no y), starting from a zero state (or from the initial state when
// they reach back to block 0) instead of from the previous CTA's hand-off.
struct JobList {
    int first, last;   // flat range [first, last) = chain * nblk + block
    int nblk;
    int cF, cL;        // first and last chain touched
    int nE, nM;        // lengths of the tail part (processed first) and of the full chains
    int a, wu;         // first output block of chain cF's segment, warm-up blocks before it
    __device__ int count() const { return last - first + wu; }
    // job J is a warm-up block (the first wu jobs of chain cF's segment, which runs last)
    __device__ __forceinline__ bool warm(int J) const {
        return wu > 0 && (cF == cL ? J < wu : (J >= nE + nM && J < nE + nM + wu));
    }
    __device__ __forceinline__ void at(int J, int& chain, int& blk, int& seg_lo, int& seg_hi) const {
        if (cF == cL) {
            chain = cF;
            seg_lo = a - wu;
            blk = seg_lo + J;
            seg_hi = last - cF * nblk;
        } else if (J < nE) {
            chain = cL;
            blk = J;
            seg_lo = 0;
            seg_hi = nE;
        } else if (J < nE + nM) {
            const unsigned r = static_cast<unsigned>(J - nE);
            chain = cF + 1 + static_cast<int>(r / static_cast<unsigned>(nblk));
            blk = static_cast<int>(r % static_cast<unsigned>(nblk));
            seg_lo = 0;
            seg_hi = nblk;
        } else {
            chain = cF;
            seg_lo = a - wu;
            blk = seg_lo + (J - nE - nM);
            seg_hi = nblk;
        }
    }
};

__device__ __forceinline__ JobList make_jobs(const ChainParams& p, int first, int last) {
    JobList jl;
    jl.first = first;
    jl.last = last;
    jl.nblk = p.nblk;
    jl.cF = jl.first / p.nblk;
    jl.cL = (jl.last - 1) / p.nblk;
    jl.nE = jl.last - jl.cL * p.nblk;
    jl.nM = (jl.cF == jl.cL) ? 0 : (jl.cL - jl.cF - 1) * p.nblk;
    jl.a = jl.first - jl.cF * p.nblk;
    jl.wu = 0;
    return jl;
}

struct JobPos {
    int blk, lo, hi;  // block, and the block range of the job's segment
    int b, cb, g;     // batch row, chain (head pair) within the row, B/C group
    int h[kHG];       // the heads of the chain's two 64-row halves (one head twice at headdim 128)
    int p0[kHG];      // the first p of each half within its head (0, or 0 and 64 at headdim 128)
    bool warm;        // warm-up block: advances the state, writes no y
    bool wait;        // the segment starts from the previous CTA's hand-off
};

__device__ __forceinline__ JobPos job_pos(const JobList& jobs, int J, int chains_per_b, int HperG,
                                       const int* __restrict__ order, uint32_t* status, int hpc = kHG) {
    JobPos jp;
    int chain;
    jobs.at(J, chain, jp.blk, jp.lo, jp.hi);
    jp.b = chain / chains_per_b;
    jp.cb = chain - jp.b * chains_per_b;
    jp.g = (jp.cb * hpc) / HperG;  // pairs never straddle a group
    if (hpc == kHG) {
        // the pair order, from this CTA's shared-memory copy (null: the natural order 2 cb, 2 cb + 1)
        jp.h[0] = order ? order[kHG * jp.cb] : kHG * jp.cb;
        jp.h[1] = order ? order[kHG * jp.cb + 1] : kHG * jp.cb + 1;
        jp.p0[0] = jp.p0[1] = 0;
    } else {  // headdim 128: chain cb is head cb, its halves p < 64 and p >= 64
        jp.h[0] = jp.h[1] = jp.cb;
        jp.p0[0] = 0;
        jp.p0[1] = kP;
    }
    // a job inside its segment and the block range; both heads real heads of the pair's group
    SSD_CHECK(status, J >= 0 && J < jobs.count() && 0 <= jp.lo && jp.lo <= jp.blk && jp.blk < jp.hi &&
                          jp.hi <= jobs.nblk && chain >= 0);
    SSD_CHECK(status, jp.h[0] >= 0 && jp.h[1] >= 0 && jp.h[0] < hpc * chains_per_b && jp.h[1] < hpc * chains_per_b &&
                          (hpc == kHG ? jp.h[0] != jp.h[1] : jp.h[0] == jp.h[1]) && jp.h[0] / HperG == jp.g &&
                          jp.h[1] / HperG == jp.g);
    const bool seg_f = (chain == jobs.cF);
    jp.warm = seg_f && jp.blk < jobs.a;
    jp.wait = seg_f && jp.lo > 0 && jobs.wu == 0;
    return jp;
}

// softplus(v) = max(v, 0) + log1p(z), z = e^{-|v|} in (0, 1]. log1p(z) is the
// Taylor series z - z^2/2 + z^3/3 - z^4/4 for z < 1/32 (truncation under
// z^5/5: a relative 2e-7) and log(1 + z) above, where the rounding of 1 + z
// (2^-24) is at most 2e-6 of the result (>= 0.03); the exponential and the
// logarithm are the fast hardware approximations (a few ulp).
__device__ __forceinline__ float softplus_f(float v) {
    const float z = __expf(-fabsf(v));
    const float l = z < 0.03125f ? z * (1.f - z * (0.5f - z * (0.33333334f - 0.25f * z))) : __logf(1.f + z);
    return fmaxf(v, 0.f) + l;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t v) {
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&v);
    return __bfloat1622float2(b);
}

// Bounded wait on this CTA's own pipeline. A timeout sets bit 1 of the status
// word and the CTA's abort flag; after that no role waits on the pipeline any
// more, so every loop runs out quickly (the results are then invalid and the
// host is told). Copies and MMAs already issued are still drained before exit.
__device__ __noinline__ void wait_bar(uint64_t* bar, uint32_t parity, uint32_t* status, volatile uint32_t* abort) {
    if (*abort) return;
    if (!ptx::mbar_wait(bar, parity, kLocalWaitNs)) {
        atomicOr(status, 2u);
        *abort = 1u;
    }
}

__device__ __forceinline__ void warp_arrive(uint64_t* bar, int lane) {
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(bar);
}

// Operand offsets (descriptor units of 16 bytes) of K step k (16 elements):
// K-major [rows][64] tiles: +32 B inside a tile, the next 64-column tile after
// four steps; MN-major tiles (rows along K): +16 rows of 128 B.
__device__ __forceinline__ uint64_t kmaj(int k) {
    return static_cast<uint64_t>((((k >> 2) * kTile + (k & 3) * 32) >> 4));
}
__device__ __forceinline__ uint64_t mnmaj(int k) { return static_cast<uint64_t>((k * 2048) >> 4); }

// k3 of one sub-block: Z += W^T B over its K steps [k0, k0 + nk).
__device__ __noinline__ void mma_k3(uint32_t z, uint64_t a_w, uint64_t b_b, uint32_t idesc, int k0, int nk) {
#pragma unroll 1
    for (int k = k0; k < k0 + nk; ++k) ptx::mma_bf16(z, a_w + mnmaj(k), b_b + mnmaj(k), idesc, 1u);
}

// k5a of one sub-block: Y^T[:, t0 : t0 + QS] = W^T L^T over s in the sub-block
// (L rows from t0, K steps [k0, k0 + nk)); the first step overwrites the columns.
__device__ __noinline__ void mma_k5a(uint32_t y, uint64_t a_w, uint64_t b_l, uint32_t idesc, int k0, int nk) {
#pragma unroll 1
    for (int k = k0; k < k0 + nk; ++k) ptx::mma_bf16(y, a_w + mnmaj(k), b_l + kmaj(k), idesc, k > k0 ? 1u : 0u);
}

// k5b of one sub-block: Y^T[:, t0 : t0 + QS] (+)= H C^T, H from TMEM (8 columns per
// step); it overwrites the columns of extreme sub-blocks, which have no k5a.
__device__ __noinline__ void mma_k5b(uint32_t y, uint32_t h_tmem, uint64_t b_c, uint32_t idesc, uint32_t acc) {
#pragma unroll 1
    for (int k = 0; k < 8; ++k) ptx::mma_bf16_ta(y, h_tmem + 8 * k, b_c + kmaj(k), idesc, (acc | k) ? 1u : 0u);
}

__device__ __forceinline__ uint32_t idesc_n(int n, bool a_mn, bool b_mn) {
    return ptx::idesc_bf16_f32(128, n, a_mn, b_mn);
}

// The rare tokens of one (head, p), out of line, rewritten in global memory
// after the tile store: in extreme sub-blocks y_t = u_t Y_t + D x_t + the
// intra-block sum over s in [s0, t] with per-entry decays (every factor
// e^{cs_t - cs_s} <= 1); elsewhere, where wf_t < kTinyWF, y_t = u_t Y_t + D x_t.
// Y comes again from TMEM, x and L from global memory, u and wf from the job's
// tables, cumsum and dt from its record in global memory.
__device__ __noinline__ void fixup_tokens(uint32_t ycol, uint32_t extreme, int qs, int tn, const float* uf,
                                          const float* wf, const float* cs, const float* dtv, float Dh,
                                          const __nv_bfloat16* xg, __nv_bfloat16* yg, long long x_tstride,
                                          const __nv_bfloat16* lg) {
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
        uint32_t r[32];
        ptx::tmem_ld32(ycol + 32 * k, r);
        // x of the chunk's rare tokens, all loads in flight at once
        uint32_t pick = 0u;
        float xv[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const int t = 32 * k + e;
            const bool on = t < tn && (((extreme >> (t / qs)) & 1u) || wf[t] < kTinyWF);
            pick |= (on ? 1u : 0u) << e;
            xv[e] = on ? __bfloat162float(xg[t * x_tstride]) : 0.f;
        }
        ptx::tmem_wait_ld(r);
        if (pick == 0u) continue;
#pragma unroll 1
        for (int e = 0; e < 32; ++e) {
            if (!((pick >> e) & 1u)) continue;
            const int t = 32 * k + e;
            float acc = fmaf(uf[t], __uint_as_float(r[e]), Dh * xv[e]);
            if ((extreme >> (t / qs)) & 1u)
                for (int s = (t / qs) * qs; s <= t; ++s)
                    acc = fmaf(__bfloat162float(lg[t * kT + s]) * __expf(cs[t] - cs[s]) * dtv[s],
                               __bfloat162float(xg[s * x_tstride]), acc);
            yg[t * x_tstride] = __float2bfloat16_rn(acc);
        }
    }
}

// This CTA's job range [first, last) when the jobs are split by estimated cost
// (all kThreads threads; out[0..1] and sh[0..15] in shared memory). CTA c
// starts after the job i whose cost interval (before, after] holds the target
// T_c, c in [1, ncta); T_c increases with c, so every such c lands on exactly
// one job. Plain split: T_c = ceil(c total / ncta). With at least kBalanceMin
// jobs per CTA, T_{c+1} - T_c >= 10 kBalanceMin - 1 exceeds any one job's cost
// (at most 110), so no range is empty. Thread t sums the costs of a contiguous
// run of the byte array, a block scan places each thread's run on the cost
// line, and the thread whose run holds a target finds its job.
//
// Long chains (horizon != null, pen[ncta] in shared memory): a CTA whose range
// starts at block a > 0 of a chain first warms up over min(a, horizon[chain])
// blocks, so the split charges each boundary that warm-up: a first pass places
// the plain boundaries and records pen[c] (10 per warm-up block) at each, and
// the second sets T_c = ceil(c (total + sum pen) / ncta) - sum_{c' < c} pen[c'],
// so that range cost plus warm-up is the same for every CTA. A charge is
// capped at half a plain share, which keeps the boundaries increasing and, with
// kBalanceMin jobs per CTA, every range non-empty.
__device__ __noinline__ void cta_range(const uint8_t* cost, long long njob, long long ncta, int cta,
                                       unsigned long long* sh, uint32_t* out, const int* horizon, int nblk,
                                       uint32_t* pen) {
    const int t = threadIdx.x, l = t & 31, wp = t >> 5;
    const long long nw = (njob + 3) / 4;  // 4-byte words (the array is padded to them)
    const long long k = (nw + kThreads - 1) / kThreads;
    const long long w0 = min(nw, t * k), w1 = min(nw, w0 + k);
    const uint32_t* cw = reinterpret_cast<const uint32_t*>(cost);
    auto word = [&](long long i) {
        uint32_t v = __ldg(cw + i);
        for (int b = 0; b < 4; ++b)
            if (4 * i + b >= njob) v &= ~(0xffu << (8 * b));
        return v;
    };
    auto bsum = [](uint32_t v) { return (v & 0xffu) + ((v >> 8) & 0xffu) + ((v >> 16) & 0xffu) + (v >> 24); };
    unsigned long long sum = 0;
    for (long long i = w0; i < w1; ++i) sum += bsum(word(i));
    unsigned long long x = sum;  // inclusive scan over the block
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (l >= o) x += y;
    }
    if (l == 31) sh[wp] = x;
    __syncthreads();
    unsigned long long before = x - sum, total = 0;
    for (int i = 0; i < kThreads / 32; ++i) {
        if (i < wp) before += sh[i];
        total += sh[i];
    }
    // the job after the one whose cost interval holds tc, or -1 when tc is not in this thread's run
    auto find = [&](unsigned long long tc) -> long long {
        if (!(before < tc && tc <= before + sum)) return -1;
        unsigned long long run = before;
        for (long long i = w0; i < w1; ++i) {
            const uint32_t v = word(i);
            for (int b = 0; b < 4; ++b) {
                run += (v >> (8 * b)) & 0xffu;
                if (run >= tc) return 4 * i + b + 1;
            }
        }
        return -1;
    };
    unsigned long long tgt[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) tgt[e] = ((cta + e) * total + ncta - 1) / ncta;
    if (horizon) {
        // pass 1: the warm-up charge at every plain boundary, recorded by the thread that finds it
        if (t == 0) pen[0] = 0u;
        if (sum > 0) {
            long long c = static_cast<long long>((before * ncta) / total);  // the first c with T_c > before is c or c + 1
            for (; c < ncta; ++c) {
                const unsigned long long tc = (c * total + ncta - 1) / ncta;
                if (c == 0 || tc <= before) continue;
                if (tc > before + sum) break;
                const long long j = find(tc);
                const long long ch = j / nblk, a = j - ch * nblk;
                const long long wu = a > 0 ? 10 * min(a, static_cast<long long>(horizon[ch])) : 0;
                pen[c] = static_cast<uint32_t>(min(wu, static_cast<long long>(total / ncta / 2)));
            }
        }
        __syncthreads();
        unsigned long long p_all = 0, p_before[2] = {0, 0};
        for (long long c = 1; c < ncta; ++c) {
            p_all += pen[c];
#pragma unroll
            for (int e = 0; e < 2; ++e)
                if (c < cta + e) p_before[e] += pen[c];
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const long long tc = static_cast<long long>(((cta + e) * (total + p_all) + ncta - 1) / ncta) -
                                 static_cast<long long>(p_before[e]);
            tgt[e] = static_cast<unsigned long long>(max(1ll, min(tc, static_cast<long long>(total))));
        }
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const long long c = cta + e;
        if (c == 0 || c == ncta) continue;
        const long long j = find(tgt[e]);
        if (j >= 0) out[e] = static_cast<uint32_t>(j);
    }
    __syncthreads();
}

// Per-chain warm-up horizon for the long-chain split (all kThreads threads):
// the mean block decay of each head over the chain, from the per-job decays;
// horizon[chain] = min(nblk, ceil(kWarmupNats / the smaller mean)) blocks.
// dsum[2 nchains] is shared-memory scratch.
__device__ __noinline__ void chain_horizons(const float2* __restrict__ decay, long long njob, int nblk, int nchains,
                                            float* dsum, int* horizon) {
    const int t = threadIdx.x;
    for (int i = t; i < 2 * nchains; i += kThreads) dsum[i] = 0.f;
    __syncthreads();
    const long long k = (njob + kThreads - 1) / kThreads;
    const long long j0 = min(njob, t * k), j1 = min(njob, j0 + k);
    long long cur = -1;
    float a0 = 0.f, a1 = 0.f;
    for (long long j = j0; j < j1; ++j) {
        const long long c = j / nblk;
        if (c != cur) {
            if (cur >= 0) {
                atomicAdd(dsum + 2 * cur, a0);
                atomicAdd(dsum + 2 * cur + 1, a1);
            }
            cur = c;
            a0 = a1 = 0.f;
        }
        const float2 d = __ldg(decay + j);
        a0 += d.x;
        a1 += d.y;
    }
    if (cur >= 0) {
        atomicAdd(dsum + 2 * cur, a0);
        atomicAdd(dsum + 2 * cur + 1, a1);
    }
    __syncthreads();
    for (int c = t; c < nchains; c += kThreads) {
        const float m = fminf(dsum[2 * c], dsum[2 * c + 1]) / static_cast<float>(nblk);
        horizon[c] = m > 0.f ? static_cast<int>(fminf(ceilf(kWarmupNats / m), static_cast<float>(nblk))) : nblk;
    }
    __syncthreads();
}

// Warm-up blocks before the segment of chain cF that starts at block a > 0 (one
// warp; 0 = take the previous CTA's hand-off). The horizon m is the number of
// blocks before a over which both heads decay by kWarmupNats (all of [0, a) if
// they never do: then the warm-up starts from the chain's initial state and is
// exact). Costs are in the job-cost units of cta_range. The hand-off is ready
// no earlier than the chain's blocks [0, a) take when run one after another
// (t_ready); this CTA needs it once the rest of its range is done (t_need, the
// segment runs last). Waiting ends the range at t_ready + t_seg, warming up at
// t_range + cost(warm-up), a warm-up block taking kWarmupCostPct percent of its
// job cost (it loads no L or C and has no k5 or epilogue): warm up when that is
// earlier (warmup = 1), or always (warmup = 2, or long chains, whose split
// already charges it). Every load of a pass over the bytes is issued before
// the first sum, so the decision costs about one memory round trip per 128
// jobs of the chain.
__device__ __noinline__ int warmup_blocks(const ChainParams& prm, const JobList& jobs, int lane, bool force) {
    const int a = jobs.a;
    const long long base = static_cast<long long>(jobs.cF) * jobs.nblk;
    // horizon: walk back from block a - 1, 32 blocks per step
    int m = a;
    float d0 = 0.f, d1 = 0.f;
    for (int k0 = a - 1; k0 >= 0; k0 -= 32) {
        const int k = k0 - lane;
        float e0 = 0.f, e1 = 0.f;
        if (k >= 0) {
            const float2 e = __ldg(prm.decay + base + k);
            e0 = e.x;
            e1 = e.y;
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {  // inclusive scan: lane l sums blocks k0 - l .. k0
            const float t0 = __shfl_up_sync(0xffffffffu, e0, o), t1 = __shfl_up_sync(0xffffffffu, e1, o);
            if (lane >= o) {
                e0 += t0;
                e1 += t1;
            }
        }
        const bool ok = k >= 0 && d0 + e0 >= kWarmupNats && d1 + e1 >= kWarmupNats;
        const uint32_t hit = __ballot_sync(0xffffffffu, ok);
        if (hit) {
            m = a - (k0 - (__ffs(hit) - 1));
            break;
        }
        d0 += __shfl_sync(0xffffffffu, e0, 31);
        d1 += __shfl_sync(0xffffffffu, e1, 31);
    }
    if (prm.warmup == 2 || force) return m;
    // one pass over the cost bytes of [base, max(last, segment end)): every job
    // byte falls into the sums it belongs to
    const long long seg_end = jobs.cF == jobs.cL ? jobs.last : base + jobs.nblk;
    const long long hi = max(static_cast<long long>(jobs.last), seg_end);
    const long long wu0 = base + a - m;
    uint32_t t_ready = 0, t_range = 0, t_seg = 0, t_wu = 0;
    for (long long j0 = base & ~3ll; j0 < hi; j0 += 128) {
        const long long j = j0 + 4 * lane;
        const uint32_t v = j < hi ? __ldg(reinterpret_cast<const uint32_t*>(prm.job_cost + j)) : 0u;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const long long q = j + e;
            const uint32_t c = (v >> (8 * e)) & 0xffu;
            if (q >= base && q < base + a) t_ready += c;
            if (q >= wu0 && q < base + a) t_wu += c;
            if (q >= jobs.first && q < jobs.last) t_range += c;
            if (q >= jobs.first && q < seg_end) t_seg += c;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        t_ready += __shfl_xor_sync(0xffffffffu, t_ready, o);
        t_wu += __shfl_xor_sync(0xffffffffu, t_wu, o);
        t_range += __shfl_xor_sync(0xffffffffu, t_range, o);
        t_seg += __shfl_xor_sync(0xffffffffu, t_seg, o);
    }
    return (t_range + (t_wu * kWarmupCostPct) / 100 < t_ready + t_seg) ? m : 0;
}

template <int NS, int PD>  // dstate, headdim
__global__ void __launch_bounds__(kThreads, 1)
    ssd_chain_fused(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_l,
                    const __grid_constant__ CUtensorMap tm_y, const ChainParams prm) {
    using K = Cfg;
    using Y = Lay<NS>;
    static_assert(PD == kP || PD == 2 * kP, "headdim 64 or 128");
    constexpr int kHpc = PD == kP ? kHG : 1;  // heads per chain
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + K::OFF_BAR);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + K::OFF_MISC);
    const uint32_t sbase = ptx::smem_u32(smem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3;  // TMEM lane quarter
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;

    auto T = [&](int slot, int j, int arr) {
        return reinterpret_cast<float*>(smem + K::OFF_TAB + slot * kRecSmem) + (j * kNumTab + arr) * kT;
    };
    auto S = [&](int slot, int j) {
        return reinterpret_cast<float*>(smem + K::OFF_TAB + slot * kRecSmem + kRecTab) + j * kScal;
    };
    auto JW = [&](int slot) {
        return reinterpret_cast<uint32_t*>(smem + K::OFF_TAB + slot * kRecSmem + kRecTab + kRecScal);
    };

    if (tid == 0) {
        misc[1] = atomicAdd(prm.ticket, 1u);
        uint32_t counts[B_COUNT];
        for (int i = 0; i < B_COUNT; ++i) counts[i] = 1;
        for (int i = 0; i < kTabSlots; ++i) counts[B_TAB_EMPTY0 + i] = 5;  // epilogue warps, k3 issuer
        for (int i = 0; i < kXWMax; ++i) {
            counts[B_W_FULL0 + i] = 4;                                      // W warps
            counts[B_XW_FREE0 + i] = 2;                                     // k3 and k5a commits
        }
        counts[B_SCALED] = 4;                                               // state warps
        counts[B_H_FULL0] = counts[B_H_FULL1] = 4;                          // state warps
        counts[B_Y_EMPTY0] = counts[B_Y_EMPTY1] = 4;                        // epilogue warps
        // B_XW_EMPTY: one epilogue thread, once the y store has read the slot
        for (int i = 0; i < B_COUNT; ++i) ptx::mbar_init(&bars[i], counts[i]);
        misc[3] = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(misc, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];
    const int cta = static_cast<int>(misc[1]);
    volatile uint32_t* abort_flag = misc + 3;
    ptx::griddep_wait();  // L tiles, tables and costs from the two kernels before
    auto WB = [&](int bar, uint32_t parity) { wait_bar(&bars[bar], parity, prm.status, abort_flag); };
    int first = static_cast<int>(prm.total * cta / prm.ncta), last = static_cast<int>(prm.total * (cta + 1) / prm.ncta);
    // Long chains (more than two CTA shares of jobs): most CTAs lie inside one
    // chain, their hand-offs would come one after another, so every CTA
    // boundary inside a chain warms up, and
    // the split charges each boundary its warm-up. The ring and X/W areas of
    // shared memory serve as scratch until the pipeline starts.
    const bool long_chains = prm.cost && prm.warmup != 0 && static_cast<long long>(prm.nblk) * prm.ncta > 2 * prm.total &&
                             static_cast<long long>(prm.nchains) * 12 + 4 * prm.ncta <= 12 * kTile;
    if (prm.cost) {
        uint32_t* out = misc + 4;
        int* horizon = nullptr;
        uint32_t* pen = nullptr;
        if (long_chains) {
            float* dsum = reinterpret_cast<float*>(smem + K::OFF_RING);
            horizon = reinterpret_cast<int*>(dsum + 2 * prm.nchains);
            pen = reinterpret_cast<uint32_t*>(horizon + prm.nchains);
            chain_horizons(prm.decay, prm.total, prm.nblk, prm.nchains, dsum, horizon);
        }
        cta_range(prm.cost, prm.total, prm.ncta, cta, reinterpret_cast<unsigned long long*>(smem + K::OFF_SCAN), out,
                  horizon, prm.nblk, pen);
        if (long_chains) {  // the scratch is overwritten by TMA copies next
            ptx::fence_proxy_async_smem();
            __syncthreads();
        }
        first = cta == 0 ? 0 : static_cast<int>(out[0]);
        last = cta == prm.ncta - 1 ? static_cast<int>(prm.total) : static_cast<int>(out[1]);
    }
    SSD_CHECK(prm.status, 0 <= first && first < last && last <= prm.total);
    JobList jobs = make_jobs(prm, first, last);
    if (jobs.a > 0 && prm.warmup != 0) {
        if (warp == 0) {
            const int wu = warmup_blocks(prm, jobs, lane, long_chains);
            if (lane == 0) misc[6] = static_cast<uint32_t>(wu);
        }
        __syncthreads();
        jobs.wu = static_cast<int>(misc[6]);
    }
    const int njobs = jobs.count();
    const int HperG = prm.H / prm.G;
    const int chains_per_b = prm.H / kHpc;
    // the pair order into shared memory: every role looks heads up per job; with
    // more heads than the prep kernel sorts, the order is the natural one
    int* order = nullptr;
    if (prm.H <= kSortMaxHeads) {
        order = reinterpret_cast<int*>(smem + K::OFF_ORDER);
        for (int i = tid; i < prm.H; i += kThreads) order[i] = __ldg(prm.order + i);
        __syncthreads();
    }

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer: L, B, C ring
        if (lane == 0) {
            // L, B and C are read again by every head pair of the group: last out of L2
            const uint64_t keep = ptx::policy_evict_last();
            const int npos = Y::kKinds * njobs;
            int pr = 0;
            for (; pr < npos; ++pr) {
                const int rs = pr % Y::kRing, ru = pr / Y::kRing;
                if (ru > 0) WB(B_R_EMPTY0 + rs, (ru - 1) & 1);
                if (*abort_flag) break;
                const int J = pr / Y::kKinds, kind = pr - Y::kKinds * J;
                const JobPos jp = job_pos(jobs, J, chains_per_b, HperG, order, prm.status, kHpc);
                uint64_t* fb = &bars[B_R_FULL0 + rs];
                uint8_t* dst = smem + K::OFF_RING + rs * 2 * kTile;
                const bool is_b = !Y::kOwnB && kind >= Y::kindB(0) && kind < Y::kindB(0) + Y::kNB;
                if (jp.warm && !is_b) {
                    // a warm-up block writes no y: no L or C, the entry's phase completes empty
                    ptx::mbar_arrive(fb);
                    continue;
                }
                ptx::mbar_arrive_expect_tx(fb, 2 * kTile);
                SSD_CHECK(prm.status, rs < Y::kRing && jp.b < prm.batch && jp.g < prm.G);
                if (kind == Y::kindL()) {
                    const int tile = (jp.b * prm.nblk + jp.blk) * prm.G + jp.g;
                    SSD_CHECK(prm.status, tile >= 0 && tile < prm.batch * prm.nblk * prm.G);
                    ptx::tma_load_4d(dst, &tm_l, fb, 0, 0, 0, tile, keep);
                    ptx::tma_load_4d(dst + kTile, &tm_l, fb, 64, 0, 0, tile, keep);
                    if (Y::kNB == 2) {
                        // the second C half loads only once k5a has freed this slot: into L2 now
                        ptx::tma_prefetch_4d(&tm_c, 128, jp.g, jp.blk * kT, jp.b);
                        ptx::tma_prefetch_4d(&tm_c, 192, jp.g, jp.blk * kT, jp.b);
                    }
                } else {
                    // a 128-column half of B or C: n in [128 half, 128 half + 128)
                    const int n0 = 128 * (is_b ? kind - Y::kindB(0) : kind - Y::kindC(0));
                    const CUtensorMap* m = is_b ? &tm_b : &tm_c;
                    // a TMA copy's innermost coordinate must stay 16-byte aligned (8 bf16)
                    SSD_CHECK(prm.status, n0 % 8 == 0 && n0 >= 0 && n0 + 128 <= NS);
                    ptx::tma_load_4d(dst, m, fb, n0, jp.g, jp.blk * kT, jp.b, keep);
                    ptx::tma_load_4d(dst + kTile, m, fb, n0 + 64, jp.g, jp.blk * kT, jp.b, keep);
                }
            }
            // no copy into shared memory may be left in flight at exit: wait for the
            // last load of each slot (earlier ones completed before their reuse)
            for (int i = 0; i < Y::kRing && i < pr; ++i) {
                const int P = pr - 1 - i;
                ptx::mbar_wait(&bars[B_R_FULL0 + P % Y::kRing], (P / Y::kRing) & 1, kLocalWaitNs);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer: k3
        if (lane == 0) {
            uint32_t u = 0;  // sub-blocks so far
            // kOwnB: B of job J into its buffer (phase J of B_B_FULL), all 2 kNB tiles
            int nb = 0;  // B loads issued
            const uint64_t keep = ptx::policy_evict_last();  // B is read again by the group's other pairs
            auto load_b = [&](int J) {
                const JobPos jp = job_pos(jobs, J, chains_per_b, HperG, order, prm.status, kHpc);
                SSD_CHECK(prm.status, jp.b < prm.batch && jp.g < prm.G);
                ptx::mbar_arrive_expect_tx(&bars[B_B_FULL], 2 * Y::kNB * kTile);
                for (int i = 0; i < 2 * Y::kNB; ++i)
                    ptx::tma_load_4d(smem + Y::OFF_B + i * kTile, &tm_b, &bars[B_B_FULL], 64 * i, jp.g, jp.blk * kT,
                                     jp.b, keep);
                ++nb;
            };
            if (Y::kOwnB && njobs > 0) load_b(0);
            for (int J = 0; J < njobs; ++J) {
                const int ts = J & (kTabSlots - 1), xs = J % Y::kXW;
                WB(B_TAB_FULL0 + ts, (J / kTabSlots) & 1);
                const int nq = static_cast<int>(JW(ts)[0]);
                const int ksub = 8 / nq;  // K steps per sub-block
                ptx::mbar_arrive(&bars[B_TAB_EMPTY0 + ts]);  // this issuer is done with the record
                WB(B_W_FULL0 + xs, (J / Y::kXW) & 1);
                const uint64_t a_w = ptx::desc_sw128(sbase + Y::OFF_XW + xs * 2 * kTile, kTile, 1024);
                uint64_t b_b[Y::kNB];
                if (Y::kOwnB) {
                    WB(B_B_FULL, J & 1);
                    b_b[0] = ptx::desc_sw128(sbase + Y::OFF_B, kTile, 1024);  // N = NS over 2 kNB tiles
                } else {
#pragma unroll
                    for (int hh = 0; hh < Y::kNB; ++hh) {
                        const int pb = Y::kKinds * J + Y::kindB(hh);
                        WB(B_R_FULL0 + pb % Y::kRing, (pb / Y::kRing) & 1);
                        b_b[hh] = ptx::desc_sw128(sbase + K::OFF_RING + (pb % Y::kRing) * 2 * kTile, kTile, 1024);
                    }
                }
                for (int q = 0; q < nq; ++q, ++u) {
                    WB(B_SCALED, u & 1);
                    ptx::tc_fence_after();
                    if (Y::kOwnB) {
                        if (SSD_CHECK(prm.status, Y::COL_Z + NS <= Y::COL_H && (q + 1) * ksub <= 8))
                            mma_k3(tmem + Y::COL_Z, a_w, b_b[0], idesc_n(NS, true, true), q * ksub, ksub);
                    } else {
#pragma unroll
                        for (int hh = 0; hh < Y::kNB; ++hh)  // Z columns [128 hh, 128 hh + 128) are n of that half
                            if (SSD_CHECK(prm.status, Y::COL_Z + 128 * hh + 128 <= Y::COL_H && (q + 1) * ksub <= 8))
                                mma_k3(tmem + Y::COL_Z + 128 * hh, a_w, b_b[hh], idesc_n(128, true, true), q * ksub,
                                       ksub);
                    }
                    ptx::mma_commit(&bars[B_S_DONE]);
                }
                if (Y::kOwnB) {
                    ptx::mma_commit(&bars[B_B_EMPTY]);
                } else {
#pragma unroll
                    for (int hh = 0; hh < Y::kNB; ++hh)
                        ptx::mma_commit(&bars[B_R_EMPTY0 + (Y::kKinds * J + Y::kindB(hh)) % Y::kRing]);
                }
                ptx::mma_commit(&bars[B_XW_FREE0 + xs]);
                if (Y::kOwnB && J + 1 < njobs) {
                    WB(B_B_EMPTY, J & 1);  // k3 of job J has read B
                    if (*abort_flag) break;
                    load_b(J + 1);
                }
            }
            // no copy into shared memory may be left in flight at exit
            if (nb > 0) ptx::mbar_wait(&bars[B_B_FULL], (nb - 1) & 1, kLocalWaitNs);
            ptx::mma_commit(&bars[B_DRAIN_K3]);
            ptx::mbar_wait(&bars[B_DRAIN_K3], 0, kLocalWaitNs);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------------ MMA issuer: k5a, k5b
        if (lane == 0) {
            uint32_t u = 0;
            for (int J = 0; J < njobs; ++J) {
                const int ts = J & (kTabSlots - 1), xs = J % Y::kXW, yb = J % Y::kYBuf;
                WB(B_TAB_FULL0 + ts, (J / kTabSlots) & 1);
                const int nq = static_cast<int>(JW(ts)[0]);
                const uint32_t extreme = JW(ts)[1];
                const int qs = kT / nq, ksub = 8 / nq;
                const uint32_t yc = tmem + Y::COL_Y + 128 * yb;
                const int pl = Y::kKinds * J + Y::kindL();
                const bool warm = jobs.warm(J);  // no output: no k5a / k5b
                if (J >= Y::kYBuf)  // the epilogue has read job J - kYBuf
                    WB(B_Y_EMPTY0 + yb, ((J / Y::kYBuf) - 1) & 1);
                WB(B_W_FULL0 + xs, (J / Y::kXW) & 1);
                WB(B_R_FULL0 + pl % Y::kRing, (pl / Y::kRing) & 1);
                ptx::tc_fence_after();
                const uint64_t a_w = ptx::desc_sw128(sbase + Y::OFF_XW + xs * 2 * kTile, kTile, 1024);
                const uint32_t id_a = idesc_n(qs, true, false), id_b = idesc_n(qs, false, false);
                for (int q = 0; q < nq && !warm; ++q) {
                    if ((extreme >> q) & 1u) continue;
                    const uint64_t b_l =
                        ptx::desc_sw128(sbase + K::OFF_RING + (pl % Y::kRing) * 2 * kTile + q * qs * 128, 16, 1024);
                    if (SSD_CHECK(prm.status, yb < Y::kYBuf && (q + 1) * qs <= kT && (q + 1) * ksub <= 8 &&
                                                  Y::COL_Y + 128 * yb + 128 <= 512))
                        mma_k5a(yc + q * qs, a_w, b_l, id_a, q * ksub, ksub);
                }
                ptx::mma_commit(&bars[B_R_EMPTY0 + pl % Y::kRing]);
                ptx::mma_commit(&bars[B_XW_FREE0 + xs]);
                // the second C half (dstate 256) is waited for only before its first k5b
                // MMAs: it loads once k5a has freed L's slot, and the first half's MMAs
                // run meanwhile
                uint32_t c_slot[Y::kNB];
                uint32_t c_have = 0u;
                auto wait_c = [&](int hh) {
                    if ((c_have >> hh) & 1u) return;
                    const int pc = Y::kKinds * J + Y::kindC(hh);
                    WB(B_R_FULL0 + pc % Y::kRing, (pc / Y::kRing) & 1);
                    c_slot[hh] = sbase + K::OFF_RING + (pc % Y::kRing) * 2 * kTile;
                    c_have |= 1u << hh;
                };
                wait_c(0);
                for (int q = 0; q < nq; ++q, ++u) {
                    const int hb = u % Y::kHBuf;
                    WB(B_H_FULL0 + hb, (u / Y::kHBuf) & 1);
                    ptx::tc_fence_after();
                    if (!warm) {
#pragma unroll
                        for (int hh = 0; hh < Y::kNB; ++hh) {  // K = n in halves: H columns 64 hh.., C half hh
                            wait_c(hh);
                            const uint64_t b_c = ptx::desc_sw128(c_slot[hh] + q * qs * 128, 16, 1024);
                            if (SSD_CHECK(prm.status, hb < Y::kHBuf && Y::COL_H + (NS / 2) * hb + 64 * hh + 64 <= Y::COL_Y &&
                                                          (q + 1) * qs <= kT))
                                mma_k5b(yc + q * qs, tmem + Y::COL_H + (NS / 2) * hb + 64 * hh, b_c, id_b,
                                        hh > 0 ? 1u : ((~extreme >> q) & 1u));
                        }
                    }
                    ptx::mma_commit(&bars[B_H_EMPTY0 + hb]);
                }
#pragma unroll
                for (int hh = 0; hh < Y::kNB; ++hh) wait_c(hh);  // warm-up jobs: the entries complete empty
#pragma unroll
                for (int hh = 0; hh < Y::kNB; ++hh)
                    ptx::mma_commit(&bars[B_R_EMPTY0 + (Y::kKinds * J + Y::kindC(hh)) % Y::kRing]);
                ptx::mma_commit(&bars[B_Y_FULL0 + yb]);
            }
            ptx::mma_commit(&bars[B_DRAIN_Y]);
            ptx::mbar_wait(&bars[B_DRAIN_Y], 0, kLocalWaitNs);
        }
        __syncwarp();
    } else if (warp == 3) {
        // ------------------------------------------------------------ TMA producer: X
        if (lane == 0) {
            const uint64_t once = ptx::policy_evict_first();  // X and the table records are read once
            int jx = 0, ntab = 0;
            for (; jx < njobs; ++jx) {
                const int ts = jx & (kTabSlots - 1);
                if (jx >= kTabSlots) WB(B_TAB_EMPTY0 + ts, ((jx / kTabSlots) - 1) & 1);
                if (*abort_flag) break;
                const JobPos jp = job_pos(jobs, jx, chains_per_b, HperG, order, prm.status, kHpc);
                const long long rec = (static_cast<long long>(jp.b) * chains_per_b + jp.cb) * prm.nblk + jp.blk;
                ptx::mbar_arrive_expect_tx(&bars[B_TAB_FULL0 + ts], kRecSmem);
                ptx::bulk_load(smem + K::OFF_TAB + ts * kRecSmem, prm.tables + rec * kRecBytes, kRecSmem,
                               &bars[B_TAB_FULL0 + ts], once);
                ++ntab;
                const int xs = jx % Y::kXW;
                if (jx >= Y::kXW) WB(B_XW_EMPTY0 + xs, ((jx / Y::kXW) - 1) & 1);  // y of job jx - kXW has left
                if (*abort_flag) break;
                uint64_t* fb = &bars[B_X_FULL0 + xs];
                uint8_t* dst = smem + Y::OFF_XW + xs * 2 * kTile;
                SSD_CHECK(prm.status, Y::OFF_XW + (xs + 1) * 2 * kTile <= K::OFF_TAB &&
                                          static_cast<long long>(jp.blk) * kT < prm.L && jp.b < prm.batch);
                ptx::mbar_arrive_expect_tx(fb, 2 * kTile);
                ptx::tma_load_4d(dst, &tm_x, fb, jp.p0[0], jp.h[0], jp.blk * kT, jp.b, once);
                ptx::tma_load_4d(dst + kTile, &tm_x, fb, jp.p0[1], jp.h[1], jp.blk * kT, jp.b, once);
                if (jp.blk == 0 && prm.init)  // a chain start: its initial states into L2 for the state warps
                    for (int j = 0; j < kHG; ++j)
                        ptx::bulk_prefetch_l2(
                            prm.init + ((static_cast<size_t>(jp.b) * prm.H + jp.h[j]) * PD + jp.p0[j]) * NS,
                            kP * NS * sizeof(float));
                if (Y::kPrefetchX && jx >= Y::kXW && jx + Y::kXW < njobs) {
                    // the X of job jx + kXW into L2: its load, once the slot is free, then hits L2
                    const JobPos jn = job_pos(jobs, jx + Y::kXW, chains_per_b, HperG, order, prm.status, kHpc);
                    ptx::tma_prefetch_4d(&tm_x, jn.p0[0], jn.h[0], jn.blk * kT, jn.b);
                    ptx::tma_prefetch_4d(&tm_x, jn.p0[1], jn.h[1], jn.blk * kT, jn.b);
                }
            }
            for (int i = 0; i < Y::kXW && i < jx; ++i) {
                const int J = jx - 1 - i;
                ptx::mbar_wait(&bars[B_X_FULL0 + J % Y::kXW], (J / Y::kXW) & 1, kLocalWaitNs);
            }

            // table copies: the last one per slot
            for (int i = 0; i < kTabSlots && i < ntab; ++i) {
                const int J = ntab - 1 - i;
                ptx::mbar_wait(&bars[B_TAB_FULL0 + (J & (kTabSlots - 1))], (J / kTabSlots) & 1, kLocalWaitNs);
            }
        }
        __syncwarp();
    } else if (warp < 8) {
        // ------------------------------------------------------------ W from X, in place
        const int wt = tid - 128;  // 0..127
        for (int J = 0; J < njobs; ++J) {
            const int ts = J & (kTabSlots - 1), xs = J % Y::kXW;
            WB(B_TAB_FULL0 + ts, (J / kTabSlots) & 1);
            WB(B_X_FULL0 + xs, (J / Y::kXW) & 1);
#pragma unroll 1
            for (int j = 0; j < kHG; ++j) {
                const float* wf = T(ts, j, TAB_WF);
                uint8_t* tile = smem + Y::OFF_XW + (xs * kHG + j) * kTile;
                // all loads first, then the stores: the compiler cannot move a load past
                // a shared-memory store it may alias
                uint4 v[8];
                float w[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int chunk = wt + 128 * i;  // 16-byte chunk; its row is chunk / 8
                    v[i] = *reinterpret_cast<const uint4*>(tile + chunk * 16);
                    w[i] = wf[chunk >> 3];
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 f0 = unpack_bf16x2(v[i].x), f1 = unpack_bf16x2(v[i].y), f2 = unpack_bf16x2(v[i].z),
                                 f3 = unpack_bf16x2(v[i].w);
                    uint4 o;
                    o.x = pack_bf16x2(f0.x * w[i], f0.y * w[i]);
                    o.y = pack_bf16x2(f1.x * w[i], f1.y * w[i]);
                    o.z = pack_bf16x2(f2.x * w[i], f2.y * w[i]);
                    o.w = pack_bf16x2(f3.x * w[i], f3.y * w[i]);
                    *reinterpret_cast<uint4*>(tile + (wt + 128 * i) * 16) = o;
                }
            }
            ptx::fence_proxy_async_smem();
            warp_arrive(&bars[B_W_FULL0 + xs], lane);
        }
    } else if (warp < 12) {
        // ------------------------------------------------------------ state
        const int st = tid - 256;    // TMEM lane = (head j, p)
        const int j = st >> 6, p = st & 63;
        float inv_prev = 1.f;        // Z = sigma s; 1 / sigma of the last sub-block
        uint32_t sdone = 0, u = 0;
        for (int J = 0; J < njobs; ++J) {
            const int ts = J & (kTabSlots - 1);
            const JobPos jp = job_pos(jobs, J, chains_per_b, HperG, order, prm.status, kHpc);
            const bool seg_start = (jp.blk == jp.lo), seg_end = (jp.blk == jp.hi - 1);
            const int h = jp.h[j];
            if (seg_start && jp.wait) {
                // wait for the previous CTA's hand-off of this chain's state
                if (st == 0) {
                    const uint32_t* f = prm.flags + (cta - 1);
                    uint32_t v = ptx::ld_acquire_gpu(f);
                    const uint64_t t0 = ptx::globaltimer_ns();
                    while (v == 0u) {
                        if (ptx::globaltimer_ns() - t0 > prm.chain_wait_ns) break;
                        __nanosleep(256);
                        v = ptx::ld_acquire_gpu(f);
                    }
                    misc[2] = (v == 0u) ? 1u : 0u;
                    if (v == 0u) atomicOr(prm.status, 1u);
                }
                ptx::named_sync(2, 128);
                ptx::fence_acquire_gpu();
            }
            WB(B_TAB_FULL0 + ts, (J / kTabSlots) & 1);
            const int nq = static_cast<int>(JW(ts)[0]);
            const float* sc = S(ts, j);
            const float* src = nullptr;  // segment start: the incoming state row [n]
            if (seg_start) {
                if (jp.wait)
                    src = misc[2] ? nullptr : prm.handoff + ((static_cast<size_t>(cta - 1) * kHG + j) * kP + p) * NS;
                else if (jp.lo > 0)
                    src = nullptr;  // warm-up from a zero state
                else if (prm.init)
                    src = prm.init + ((static_cast<size_t>(jp.b) * prm.H + h) * PD + jp.p0[j] + p) * NS;
                // a hand-off row of the previous CTA or an initial-state row of a real (batch, head)
                if (!SSD_CHECK(prm.status, (jp.wait ? (cta >= 1 && cta <= prm.ncta - 1)
                                                    : (jp.b < prm.batch && h >= 0 && h < prm.H)) && p < kP))
                    src = nullptr;
                // every line of the row on its way to L2 before the first load waits
                if (src)
#pragma unroll
                    for (int k = 0; k < NS / 32; ++k) ptx::prefetch_l2(src + 32 * k);
                inv_prev = 1.f;
            }
            for (int q = 0; q < nq; ++q, ++u) {
                const bool from_src = seg_start && q == 0;
                if (!from_src) {
                    WB(B_S_DONE, sdone & 1);
                    ++sdone;
                }
                const int hb = u % Y::kHBuf;
                if (u >= static_cast<uint32_t>(Y::kHBuf)) WB(B_H_EMPTY0 + hb, ((u / Y::kHBuf) - 1) & 1);
                ptx::tc_fence_after();
                const float ec = sc[SC_EC + q], hs = sc[SC_HS + q];
                const uint32_t zcol = tmem + lane_base + Y::COL_Z;
                const uint32_t hcol = tmem + lane_base + Y::COL_H + (NS / 2) * hb;
                SSD_CHECK(prm.status, hb < Y::kHBuf && Y::COL_H + (NS / 2) * (hb + 1) <= Y::COL_Y && q < 8 && ts < kTabSlots);
#pragma unroll 1
                for (int k = 0; k < NS / 32; ++k) {
                    uint32_t r[32];
                    if (from_src) {
                        if (src) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float4 v = *reinterpret_cast<const float4*>(src + 32 * k + 4 * e);
                                r[4 * e] = __float_as_uint(v.x);
                                r[4 * e + 1] = __float_as_uint(v.y);
                                r[4 * e + 2] = __float_as_uint(v.z);
                                r[4 * e + 3] = __float_as_uint(v.w);
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; ++e) r[e] = 0u;
                        }
                    } else {
                        ptx::tmem_ld32(zcol + 32 * k, r);
                        ptx::tmem_wait_ld(r);
                    }
                    // s = Z / sigma_prev is the true state; the two factors of the new
                    // scale are applied one after the other (their product can leave
                    // the fp32 range when consecutive sub-blocks both decay strongly)
                    uint32_t hp[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float s0 = __uint_as_float(r[2 * e]) * inv_prev;
                        const float s1 = __uint_as_float(r[2 * e + 1]) * inv_prev;
                        hp[e] = pack_bf16x2(s0 * hs, s1 * hs);
                        r[2 * e] = __float_as_uint(s0 * ec);
                        r[2 * e + 1] = __float_as_uint(s1 * ec);
                    }
                    ptx::tmem_st32(zcol + 32 * k, r);
                    ptx::tmem_st16(hcol + 16 * k, hp);
                }
                inv_prev = sc[SC_IS + q];
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                warp_arrive(&bars[B_SCALED], lane);
                warp_arrive(&bars[B_H_FULL0 + hb], lane);
            }
            if (seg_end) {
                // the chain's state after this block: final state, or the hand-off to CTA + 1
                const bool to_final = (jp.hi == prm.nblk);
                WB(B_S_DONE, sdone & 1);
                ++sdone;
                ptx::tc_fence_after();
                float* dst = to_final ? (prm.final_state
                                             ? prm.final_state + ((static_cast<size_t>(jp.b) * prm.H + h) * PD + jp.p0[j] + p) * NS
                                             : nullptr)
                                      : prm.handoff + ((static_cast<size_t>(cta) * kHG + j) * kP + p) * NS;
                // the final state of a real (batch, head), or this CTA's own hand-off slot
                if (!SSD_CHECK(prm.status, to_final ? (jp.b < prm.batch && h >= 0 && h < prm.H) : (cta < prm.ncta - 1)))
                    dst = nullptr;
#pragma unroll 1
                for (int k = 0; k < NS / 32; ++k) {
                    uint32_t r[32];
                    ptx::tmem_ld32(tmem + lane_base + Y::COL_Z + 32 * k, r);
                    ptx::tmem_wait_ld(r);
                    if (dst) {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            *reinterpret_cast<float4*>(dst + 32 * k + 4 * e) =
                                make_float4(__uint_as_float(r[4 * e]) * inv_prev, __uint_as_float(r[4 * e + 1]) * inv_prev,
                                            __uint_as_float(r[4 * e + 2]) * inv_prev,
                                            __uint_as_float(r[4 * e + 3]) * inv_prev);
                    }
                }
                ptx::tc_fence_before();
                if (!to_final) {
                    __threadfence();
                    ptx::named_sync(2, 128);
                    if (st == 0) ptx::st_release_gpu(prm.flags + cta, 1u);
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Warp q4 owns TMEM lanes 32 q4 .. 32 q4 + 31: head j = q4 / 2, p in
        // [32 (q4 % 2), +32), taken as two halves of 16 lanes. Y is read in the
        // 16x256b fragment layout (a thread holds token pairs of two p), W in the
        // same layout by ldmatrix.trans from the job's W tile, and
        // y = u Y + (D / wf) W goes back over W by stmatrix.trans; the two tiles
        // then leave by TMA stores and the slot is handed back to the X producer.
        const int et = tid - 384;
        const int j = q4 >> 1;
        const int lq = lane & 3;  // token pair of the thread within an 8-token group
        // ldmatrix / stmatrix row addresses: lane l serves row l % 8 of matrix l / 8
        // (matrix m: tokens + 8 (m >> 1), p chunk + (m & 1))
        const int mrow = lane & 7, mm = lane >> 3;
        const long long x_tstride = static_cast<long long>(prm.H) * PD;
        for (int J = 0; J < njobs; ++J) {
            const int ts = J & (kTabSlots - 1), yb = J % Y::kYBuf, xs = J % Y::kXW;
            WB(B_TAB_FULL0 + ts, (J / kTabSlots) & 1);
            const float2* u2 = reinterpret_cast<const float2*>(T(ts, j, TAB_U));
            const float2* g2 = reinterpret_cast<const float2*>(T(ts, j, TAB_UG));
            const uint32_t extreme = JW(ts)[1];
            const bool rare = (extreme | JW(ts)[2]) != 0u;
            const JobPos jp = job_pos(jobs, J, chains_per_b, HperG, order, prm.status, kHpc);
            WB(B_Y_FULL0 + yb, (J / Y::kYBuf) & 1);
            WB(B_XW_FREE0 + xs, (J / Y::kXW) & 1);  // k3 and k5a no longer read W
            ptx::tc_fence_after();
            if (jp.warm) {
                // a warm-up block has no output: hand the accumulator, the slot and the
                // table record straight back
                warp_arrive(&bars[B_Y_EMPTY0 + yb], lane);
                if (et == 0) ptx::mbar_arrive(&bars[B_XW_EMPTY0 + xs]);
                warp_arrive(&bars[B_TAB_EMPTY0 + ts], lane);
                continue;
            }
            const uint32_t tile = sbase + Y::OFF_XW + (xs * kHG + j) * kTile;
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
                const uint32_t ylane = tmem + (static_cast<uint32_t>(32 * q4 + 16 * hf) << 16) + Y::COL_Y + 128 * yb;
                SSD_CHECK(prm.status, yb < Y::kYBuf && Y::COL_Y + 128 * (yb + 1) <= 512 && xs < Y::kXW);
                const uint32_t pc = 4 * (q4 & 1) + 2 * hf + (mm & 1);  // 16-byte chunk of p in the row
#pragma unroll 1
                for (int k = 0; k < 4; ++k) {
                    uint32_t r[16];
                    ptx::tmem_ld16x256_x4(ylane + 32 * k, r);
                    // the W fragments and the factors of these 32 tokens while the TMEM load runs
                    uint32_t w[2][4], addr[2];
                    float2 uf[4], gf[4];
#pragma unroll
                    for (int c = 0; c < 2; ++c) {  // 16 tokens: groups g = 2c, 2c + 1
                        const int tb = 32 * k + 16 * c;
                        const int trow = tb + 8 * (mm >> 1) + mrow;
                        addr[c] = tile + trow * 128 + ((pc ^ (trow & 7)) << 4);
                        SSD_CHECK(prm.status, trow < kT && pc < 8);
                        ptx::ldmatrix_x4_trans(addr[c], w[c]);
#pragma unroll
                        for (int gg = 0; gg < 2; ++gg) {
                            const int tp = (tb + 8 * gg) / 2 + lq;  // token pair (t, t + 1) / 2
                            uf[2 * c + gg] = u2[tp];
                            gf[2 * c + gg] = g2[tp];
                        }
                    }
                    ptx::tmem_wait_ld(r);
                    if (hf == 1 && k == 3 && !rare) {
                        ptx::tc_fence_before();
                        warp_arrive(&bars[B_Y_EMPTY0 + yb], lane);  // the accumulator has been read
                    }
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t o[4];
#pragma unroll
                        for (int gg = 0; gg < 2; ++gg) {
                            const int g = 2 * c + gg;
                            const float2 u = uf[g], gw = gf[g];
#pragma unroll
                            for (int hp = 0; hp < 2; ++hp) {  // p = lr, p = 8 + lr
                                const float2 wv = unpack_bf16x2(w[c][2 * gg + hp]);
                                o[2 * gg + hp] = pack_bf16x2(fmaf(u.x, __uint_as_float(r[4 * g + 2 * hp]), gw.x * wv.x),
                                                             fmaf(u.y, __uint_as_float(r[4 * g + 2 * hp + 1]), gw.y * wv.y));
                            }
                        }
                        ptx::stmatrix_x4_trans(addr[c], o);
                    }
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::named_sync(3, 128);
            // a store starts at non-negative coordinates inside the tensor (rows past L are dropped)
            SSD_CHECK(prm.status, jp.h[0] < prm.H && jp.h[1] < prm.H && jp.b < prm.batch &&
                                      static_cast<long long>(jp.blk) * kT < prm.L);
            if (et == 0) {
                const uint64_t once = ptx::policy_evict_first();  // y is written once
                for (int jj = 0; jj < kHG; ++jj)
                    ptx::tma_store_4d(&tm_y, smem + Y::OFF_XW + (xs * kHG + jj) * kTile, jp.p0[jj], jp.h[jj],
                                      jp.blk * kT, jp.b, once);
                ptx::bulk_commit_group();
                ptx::bulk_wait_group_read0();
                ptx::mbar_arrive(&bars[B_XW_EMPTY0 + xs]);  // the slot may take the next X
            }
            if (rare) {
                // extreme sub-blocks and tokens with a tiny W factor: rewrite them in
                // global memory once the tile store has landed
                if (et == 0) {
                    ptx::bulk_wait_group0();
                    ptx::fence_proxy_async_global();
                }
                ptx::named_sync(3, 128);
                const int p = et & 63;
                const long long t0 = static_cast<long long>(jp.blk) * kT;
                const int tn = static_cast<int>(min(static_cast<long long>(kT), prm.L - t0));  // valid tokens
                SSD_CHECK(prm.status, tn >= 1 && tn <= kT && p < kP && ts < kTabSlots);
                const long long off = ((static_cast<long long>(jp.b) * prm.L + t0) * prm.H + jp.h[j]) * PD + jp.p0[j] + p;
                const long long rec = (static_cast<long long>(jp.b) * chains_per_b + jp.cb) * prm.nblk + jp.blk;
                const float* xt = reinterpret_cast<const float*>(prm.tables + rec * kRecBytes + kRecSmem) +
                                  j * kNumTabX * kT;
                const __nv_bfloat16* lg =
                    prm.masks + static_cast<size_t>((jp.b * prm.nblk + jp.blk) * prm.G + jp.g) * kT * kT;
                fixup_tokens(tmem + lane_base + Y::COL_Y + 128 * yb, extreme, kT / static_cast<int>(JW(ts)[0]), tn,
                             T(ts, j, TAB_U), T(ts, j, TAB_WF), xt + TABX_CS * kT, xt + TABX_DT * kT, S(ts, j)[SC_D],
                             prm.x + off, prm.y + off, x_tstride, lg);
                ptx::tc_fence_before();
                warp_arrive(&bars[B_Y_EMPTY0 + yb], lane);
            }
            warp_arrive(&bars[B_TAB_EMPTY0 + ts], lane);
        }
        if (et == 0) ptx::bulk_wait_group0();  // y is in global memory before the CTA exits
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 0) ptx::tmem_dealloc(tmem, 512);
}

struct TableParams {
    const float* dt;
    const float* dt_bias;
    const float* A;
    const float* D;
    uint8_t* out;      // [chain * nblk + block] table records
    uint8_t* cost;       // [jobs] estimated job costs (cta_range)
    float2* decay;       // [jobs] decay of the whole block per head (warm-up horizon)
    uint32_t* counters;  // the chain kernel's ticket and flags, zeroed here
    int ncounters;
    uint32_t* status;    // device status word (debug-build checks)
    int* order;          // [H] heads in pair order (written by CTA 0)
    const int32_t* seq;  // [batch, L] packed-sequence ids, or null
    int sort_pairs;      // pair the heads of each group by decay rate (else 2 cb, 2 cb + 1)
    int hpc;             // heads per chain: 2, or 1 at headdim 128 (both halves of chain cb are head cb)
    int jobs_per_warp;   // consecutive jobs per warp (1 or 2)
    long long L;
    int H, G, nblk, chains_per_b, total;
    float dt_min, dt_max;
};

// Estimated cost of a job in the chain kernel, in units of a tenth of a
// whole-block job: a regression of measured per-job periods on the 2.7B shape
// on the job mix puts a job split in two sub-blocks at 1.3 and one split in four
// at 1.9 whole-block jobs; eight sub-blocks, extreme sub-blocks (CUDA-core
// intra-block sum) and the tiny-W fix-up pass are weighted by their extra state
// round trips and work. At most 10 + 32 + 64 + 4 = 110.
__device__ __forceinline__ uint32_t job_cost(int nq, uint32_t extreme, int tiny) {
    const uint32_t split = nq == 2 ? 3u : nq == 4 ? 9u : nq == 8 ? 32u : 0u;
    return 10u + split + 8u * static_cast<uint32_t>(__popc(extreme)) + (tiny ? 4u : 0u);
}

constexpr int kBalanceMin = 20;  // cost balancing from this many jobs per chain CTA up (see cta_range)
constexpr int kTableWarps = 4;   // chain_tables: warps per CTA
constexpr int kTableCtasPerSm = 9;  // chain_tables: resident CTAs per SM (56 registers)

// The table record of one job: the work of one warp (see chain_tables).
__device__ __forceinline__ void table_job(const TableParams& prm, int job, int wl, const int* s_order) {
    const int blk = job % prm.nblk;
    const int chain = job / prm.nblk;
    const int b = chain / prm.chains_per_b, cb = chain % prm.chains_per_b;
    // heads per chain hpc = 2: ranks 2 cb, 2 cb + 1 of the pair order (or heads 2 cb, 2 cb + 1);
    // hpc = 1 (headdim 128): head cb for both 64-row halves
    const int c0 = prm.hpc * cb;
    const int hh[kHG] = {prm.sort_pairs ? s_order[c0] : c0, prm.sort_pairs ? s_order[c0 + 1] : c0 + prm.hpc - 1};
    SSD_CHECK(prm.status, hh[0] >= 0 && hh[1] >= 0 && hh[0] < prm.H && hh[1] < prm.H &&
                              (prm.hpc == kHG) == (hh[0] != hh[1]));
    uint8_t* rec = prm.out + static_cast<size_t>(job) * kRecBytes;
    float* tabs = reinterpret_cast<float*>(rec);
    float* scal = reinterpret_cast<float*>(rec + kRecTab);
    uint32_t* jw = reinterpret_cast<uint32_t*>(rec + kRecTab + kRecScal);
    float* tabx = reinterpret_cast<float*>(rec + kRecSmem);
    auto T = [&](int j, int arr) { return reinterpret_cast<float4*>(tabs + (j * kNumTab + arr) * kT) + wl; };
    auto TX = [&](int j, int arr) { return reinterpret_cast<float4*>(tabx + (j * kNumTabX + arr) * kT) + wl; };
    auto S = [&](int j) { return scal + j * kScal; };
    // lane wl owns tokens 4 wl .. 4 wl + 3 of the block (one 16-token unit); every
    // global load is issued here, before the first store
    const int tg0 = blk * kT + 4 * wl;
    const float2 bias = make_float2(__ldg(prm.dt_bias + hh[0]), __ldg(prm.dt_bias + hh[1]));
    const float2 a2 = make_float2(__ldg(prm.A + hh[0]), __ldg(prm.A + hh[1]));
    const float2 d2 = prm.D ? make_float2(__ldg(prm.D + hh[0]), __ldg(prm.D + hh[1])) : make_float2(0.f, 0.f);
    float2 raw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float* row = prm.dt + (static_cast<long long>(b) * prm.L + (tg0 + i)) * prm.H;
        raw[i] = tg0 + i < prm.L ? make_float2(__ldg(row + hh[0]), __ldg(row + hh[1])) : make_float2(0.f, 0.f);
    }
    float dtv[kHG][4], cs[kHG][4];
    float cut[4];  // a new packed sequence starts at the token: no state crosses (kSeqCutNats)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const long long t = tg0 + i;
        cut[i] = (prm.seq && t > 0 && t < prm.L &&
                  __ldg(prm.seq + static_cast<long long>(b) * prm.L + t) !=
                      __ldg(prm.seq + static_cast<long long>(b) * prm.L + t - 1))
                     ? -kSeqCutNats
                     : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < kHG; ++j)
            dtv[j][i] = tg0 + i < prm.L
                            ? fminf(fmaxf(softplus_f((j ? raw[i].y : raw[i].x) + (j ? bias.y : bias.x)), prm.dt_min),
                                    prm.dt_max)
                            : 0.f;
    float bnd[kHG][8];  // cumsum at token 16k + 15
    float vtot[kHG];     // cumsum at token 4 wl + 3 (this lane's last token)
#pragma unroll
    for (int j = 0; j < kHG; ++j) {
        const float a = j ? a2.y : a2.x;
        float run = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            run += fmaf(dtv[j][i], a, cut[i]);
            cs[j][i] = run;
        }
        float v = run;  // inclusive scan of the lane totals
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_up_sync(0xffffffffu, v, off);
            if (wl >= off) v += o;
        }
        const float pre = v - run;
#pragma unroll
        for (int i = 0; i < 4; ++i) cs[j][i] += pre;
        vtot[j] = v;
#pragma unroll
        for (int k = 0; k < 8; ++k) bnd[j][k] = __shfl_sync(0xffffffffu, v, 4 * k + 3);
    }
    int nq = 8;
#pragma unroll
    for (int cand = 1; cand < 8; cand <<= 1) {
        const int m = 8 / cand;  // 16-token units per sub-block
        bool ok = true;
#pragma unroll
        for (int j = 0; j < kHG; ++j)
#pragma unroll
            for (int r = 0; r < cand; ++r) {
                const float lo_ = r > 0 ? bnd[j][r * m - 1] : 0.f;
                ok = ok && (lo_ - bnd[j][(r + 1) * m - 1] <= kMaxSubDecay);
            }
        if (ok && nq == 8) nq = cand;
    }
    uint32_t extreme = 0u;
    if (nq == 8) {
#pragma unroll
        for (int j = 0; j < kHG; ++j)
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float lo_ = r > 0 ? bnd[j][r - 1] : 0.f;
                if (lo_ - bnd[j][r] > kMaxSubDecay) extreme |= 1u << r;
            }
    }
    const int qs = kT / nq;
    const int q = 4 * wl / qs;  // the lane's sub-block
    const bool ext = (extreme >> q) & 1u;
    bool any_tiny = false;
#pragma unroll
    for (int j = 0; j < kHG; ++j) {
        const float Dh = j ? d2.y : d2.x;
        // cumsum relative to the sub-block start, and the sub-block's end value: the
        // cumsums at tokens q qs - 1 and (q + 1) qs - 1 sit in lanes q qs / 4 - 1 and
        // (q + 1) qs / 4 - 1; the same shuffles give lane wl the bounds of sub-block wl
        const int ql = q * qs / 4, wlo = wl * qs / 4;
        const float sb = __shfl_sync(0xffffffffu, vtot[j], max(ql - 1, 0));
        const float se_ = __shfl_sync(0xffffffffu, vtot[j], min(ql + qs / 4, 32) - 1);
        const float lo_w = __shfl_sync(0xffffffffu, vtot[j], min(max(wlo - 1, 0), 31));
        const float hi_w = __shfl_sync(0xffffffffu, vtot[j], min(wlo + qs / 4, 32) - 1);
        const float base = q > 0 ? sb : 0.f, endv = se_;
        const float cse = endv - base;
        const float c = (-cse <= kMaxSubDecay) ? 0.5f * cse : cse + kExtremeRef;
        float wf4[4], u4[4], g4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float csl = cs[j][i] - base;
            const float e = __expf(c - csl);  // within e^{+-75} outside extreme sub-blocks
            const float wfv = dtv[j][i] * e;
            const bool tiny = !ext && wfv < kTinyWF;  // D x from x itself (fixup_tokens)
            any_tiny |= tiny && (tg0 + i < prm.L);
            wf4[i] = wfv;
            u4[i] = __expf(ext ? csl : csl - c);
            g4[i] = (ext || tiny) ? 0.f : __fdividef(Dh, wfv);
            cs[j][i] = csl;  // kept for the rare-token arrays below
        }
        *T(j, TAB_WF) = make_float4(wf4[0], wf4[1], wf4[2], wf4[3]);
        *T(j, TAB_U) = make_float4(u4[0], u4[1], u4[2], u4[3]);
        *T(j, TAB_UG) = make_float4(g4[0], g4[1], g4[2], g4[3]);
        if (wl < nq) {
            // the sub-block scalars: lane wl serves sub-block wl
            const float se = hi_w - (wl > 0 ? lo_w : 0.f);
            const bool sext = (extreme >> wl) & 1u;
            const float sc_ = (-se <= kMaxSubDecay) ? 0.5f * se : se + kExtremeRef;
            S(j)[SC_EC + wl] = __expf(sc_);
            S(j)[SC_HS + wl] = sext ? 1.f : __expf(sc_);
            S(j)[SC_IS + wl] = __expf(se - sc_);
        }
        if (wl == 0) S(j)[SC_D] = Dh;
    }
    any_tiny = __any_sync(0xffffffffu, any_tiny);
    if (extreme != 0u || any_tiny) {
        // sub-block cumsum and dt: read only by fixup_tokens, for jobs with rare tokens
#pragma unroll
        for (int j = 0; j < kHG; ++j) {
            *TX(j, TABX_CS) = make_float4(cs[j][0], cs[j][1], cs[j][2], cs[j][3]);
            *TX(j, TABX_DT) = make_float4(dtv[j][0], dtv[j][1], dtv[j][2], dtv[j][3]);
        }
    }
    if (wl == 0) {
        jw[0] = static_cast<uint32_t>(nq);
        jw[1] = extreme;
        jw[2] = any_tiny ? 1u : 0u;  // some valid token has wf < kTinyWF
        jw[3] = 0u;
        prm.cost[job] = static_cast<uint8_t>(job_cost(nq, extreme, any_tiny));
        prm.decay[job] = make_float2(-bnd[0][7], -bnd[1][7]);  // cumsum at the block's last token
    }
}

// The table record of one job (one block of one head pair), one warp per job
// (two consecutive jobs per warp where one per warp would take more than one
// wave of CTAs: every CTA ranks the heads, once for all of its jobs):
// lane l owns tokens 4l .. 4l + 3 of the block for both heads. dt =
// clamp(softplus(dt_raw + dt_bias)), the block cumsum of dt*A, the sub-block
// split (the largest of 128, 64, 32, 16 tokens whose decays all stay within
// kMaxSubDecay; 16-token sub-blocks beyond it are extreme), then per token the
// W factor, the epilogue factors u and D / wf, the sub-block-relative cumsum
// and dt, and per sub-block the state scales e^{c}, the H scale and 1 / sigma;
// besides the record, the job's cost and its block decay per head (the warm-up horizon).
//
// Head pairs: within each B/C group the heads are ranked by their decay rate
// clamp(softplus(dt_bias)) * (-A) and paired rank 2i with rank 2i + 1, so that
// fast-decaying heads (whose blocks split into sub-blocks) share chains and a
// slowly decaying head is not tied to them. Every CTA ranks the heads itself
// (nheads x heads-per-group comparisons); CTA 0 also stores the order for the
// chain kernel. The pairing only schedules: each head's result is its own.
// At most 56 registers so that 9 CTAs fit an SM: the 1280 CTAs of the 2.7B shape in one wave.
__global__ void __launch_bounds__(kTableWarps * 32, kTableCtasPerSm) chain_tables(const TableParams prm) {
    __shared__ __align__(16) uint32_t s_key[kSortMaxHeads];
    __shared__ int s_order[kSortMaxHeads];
    // launched early behind the previous kernel of the stream (which may still use the
    // workspace or write the inputs): nothing is touched before it completes
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();  // chain_masks does not read the tables until its end
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < prm.ncounters; i += blockDim.x) prm.counters[i] = 0u;
    if (prm.sort_pairs) {
        const int r = prm.H / prm.G;
        for (int h = threadIdx.x; h < prm.H; h += blockDim.x) {
            const float sp = fminf(fmaxf(softplus_f(__ldg(prm.dt_bias + h)), prm.dt_min), prm.dt_max);
            float k = sp * -__ldg(prm.A + h);
            k = (k == k) ? k + 0.f : __int_as_float(0x7f800000);  // NaN ranks as +inf, -0 as +0
            // the float order as an unsigned order: flip all bits of negatives, the sign of the rest
            const uint32_t u = __float_as_uint(k);
            s_key[h] = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
        }
        __syncthreads();
        // rank of head h in its group by (key, head), a strict total order: heads
        // before h count when their key is not above h's, heads after h when below
        for (int h = threadIdx.x; h < prm.H; h += blockDim.x) {
            const int g0 = (h / r) * r;
            const uint32_t kh = s_key[h];
            int rank = 0;
            for (int i = g0; i < h; ++i) rank += s_key[i] <= kh ? 1 : 0;
            for (int i = h + 1; i < g0 + r; ++i) rank += s_key[i] < kh ? 1 : 0;
            s_order[g0 + rank] = h;
        }
        __syncthreads();
    }
    if (blockIdx.x == 0)
        for (int h = threadIdx.x; h < prm.H; h += blockDim.x) prm.order[h] = prm.sort_pairs ? s_order[h] : h;
    const int wl = threadIdx.x & 31;
    // jobs_per_warp consecutive jobs per warp, one after another (job indices fit
    // 31 bits: the host launches only then)
    const int job0 = (static_cast<int>(blockIdx.x) * kTableWarps + static_cast<int>(threadIdx.x >> 5)) * prm.jobs_per_warp;
#pragma unroll 1
    for (int job = job0; job < job0 + prm.jobs_per_warp && job < prm.total; ++job) table_job(prm, job, wl, s_order);
}

// L = C.B^T masked to s <= t, in bf16, for one (batch, block, group): the matrix
// every head of the group shares (burn-mamba k2_ssd_bmm plus the causal mask),
// the contraction over all NS columns of n. One CTA of 128 threads per tile;
// thread t writes row t.
template <int NS>
constexpr uint32_t mask_smem() {
    return 2 * (NS / 64) * kTile + 64 + 1024;
}

template <int NS>
__global__ void __launch_bounds__(128)
    chain_masks(const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_c,
                __nv_bfloat16* __restrict__ out, int nblk, int G, uint32_t* status) {
    constexpr int kNT = NS / 64;  // 64-column tiles of C (and of B)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * kNT * kTile);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + 2 * kNT * kTile + 16);
    const int tile = blockIdx.x;
    const int g = tile % G, blk = (tile / G) % nblk, b = tile / (G * nblk);
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        ptx::mbar_init(&bars[0], 1);
        ptx::mbar_init(&bars[1], 1);
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(misc, 128);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];
    const uint32_t sbase = ptx::smem_u32(smem);
    if (tid == 0) {
        ptx::mbar_arrive_expect_tx(&bars[0], 2 * kNT * kTile);
        for (int i = 0; i < kNT; ++i) {
            ptx::tma_load_4d(smem + i * kTile, &tm_c, &bars[0], 64 * i, g, blk * kT, b);
            ptx::tma_load_4d(smem + (kNT + i) * kTile, &tm_b, &bars[0], 64 * i, g, blk * kT, b);
        }
        if (ptx::mbar_wait(&bars[0], 0, kLocalWaitNs)) {
            ptx::tc_fence_after();
            const uint64_t a = ptx::desc_sw128(sbase, 16, 1024),
                           bb = ptx::desc_sw128(sbase + kNT * kTile, 16, 1024);
            const uint32_t idesc = ptx::idesc_bf16_f32(128, 128, false, false);
            for (int k = 0; k < NS / 16; ++k) ptx::mma_bf16(tmem, a + kmaj(k), bb + kmaj(k), idesc, k > 0 ? 1u : 0u);
        } else {
            atomicOr(status, 2u);
        }
        ptx::mma_commit(&bars[1]);  // arrives once the MMAs (if any) complete
    }
    __syncwarp();
    if (!ptx::mbar_wait(&bars[1], 0, kLocalWaitNs)) atomicOr(status, 2u);
    ptx::tc_fence_after();
    const int t = tid;
    __nv_bfloat16* row = out + (static_cast<size_t>(tile) * kT + t) * kT;
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
        uint32_t r[32];
        ptx::tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 32 * k, r);
        ptx::tmem_wait_ld(r);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int s = 32 * k + 2 * e;
            pk[e] = pack_bf16x2(s <= t ? __uint_as_float(r[2 * e]) : 0.f,
                                s + 1 <= t ? __uint_as_float(r[2 * e + 1]) : 0.f);
        }
#pragma unroll
        for (int v = 0; v < 4; ++v)
            *reinterpret_cast<uint4*>(row + 32 * k + 8 * v) =
                make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 0) ptx::tmem_dealloc(tmem, 128);
    // this grid may overlap chain_tables, but completes only after it, so the
    // chain kernel's wait on this grid covers both; the chain kernel may launch
    // once every CTA here is past this point (no table CTA is left to schedule)
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
}

// ---------------------------------------------------------------- host side
int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

struct ChainPlan {
    int ncta;
    long long nchains, nblk, total, ntiles, nheads, ns;
};

ChainPlan plan(const ssd_dims& d, int nsm) {
    ChainPlan p;
    p.nblk = (d.seqlen + kT - 1) / kT;
    p.nchains = d.batch * d.nheads / (d.headdim == 2 * kP ? 1 : kHG);
    p.total = p.nchains * p.nblk;
    p.ncta = static_cast<int>(std::min<long long>(nsm, p.total));
    p.ntiles = d.batch * p.nblk * d.ngroups;
    p.nheads = d.nheads;
    p.ns = d.dstate;
    return p;
}

// ticket, flags [ncta]
size_t counters_bytes(int ncta) {
    return align_up(sizeof(uint32_t) * (1 + static_cast<size_t>(ncta)), kWorkspaceAlign);
}
size_t handoff_bytes(int ncta, long long ns) {
    return align_up(static_cast<size_t>(ncta) * kHG * kP * ns * sizeof(float), kWorkspaceAlign);
}
size_t masks_bytes(long long ntiles) { return align_up(static_cast<size_t>(ntiles) * kT * kT * 2, kWorkspaceAlign); }
size_t tables_bytes(long long jobs) { return align_up(static_cast<size_t>(jobs) * kRecBytes, kWorkspaceAlign); }
size_t costs_bytes(long long jobs) { return align_up(static_cast<size_t>(jobs), kWorkspaceAlign); }
size_t order_bytes(long long heads) { return align_up(static_cast<size_t>(heads) * sizeof(int), kWorkspaceAlign); }
size_t decay_bytes(long long jobs) { return align_up(static_cast<size_t>(jobs) * sizeof(float2), kWorkspaceAlign); }
size_t chain_ws_bytes(const ChainPlan& pl) {
    return counters_bytes(pl.ncta) + handoff_bytes(pl.ncta, pl.ns) + masks_bytes(pl.ntiles) + tables_bytes(pl.total) +
           costs_bytes(pl.total) + order_bytes(pl.nheads) + decay_bytes(pl.total);
}

template <int NS>
ssd_status launch_chain(const FwdArgs& a, void* ws, const ChainPlan& pl) {
    const ssd_dims& d = a.d;
    const size_t counters = counters_bytes(pl.ncta);
    float* handoff = reinterpret_cast<float*>(static_cast<char*>(ws) + counters);
    __nv_bfloat16* masks =
        reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(ws) + counters + handoff_bytes(pl.ncta, pl.ns));
    uint8_t* tables =
        static_cast<uint8_t*>(ws) + counters + handoff_bytes(pl.ncta, pl.ns) + masks_bytes(pl.ntiles);
    uint8_t* costs = tables + tables_bytes(pl.total);
    int* order = reinterpret_cast<int*>(costs + costs_bytes(pl.total));
    float2* decay = reinterpret_cast<float2*>(reinterpret_cast<char*>(order) + order_bytes(pl.nheads));
    CUtensorMap tx, tb, tc, tl, ty;
    if (!make_map_bf16(&tx, a.x, d.headdim, d.nheads, d.seqlen, d.batch) ||
        !make_map_bf16(&tb, a.B, d.dstate, d.ngroups, d.seqlen, d.batch) ||
        !make_map_bf16(&tc, a.C, d.dstate, d.ngroups, d.seqlen, d.batch) ||
        !make_map_bf16(&tl, masks, kT, 1, kT, static_cast<uint64_t>(pl.ntiles)) ||
        !make_map_bf16(&ty, a.y, d.headdim, d.nheads, d.seqlen, d.batch))
        return SSD_ERR_CUDA;
    if (cudaFuncSetAttribute(chain_masks<NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(mask_smem<NS>())) != cudaSuccess)
        return SSD_ERR_CUDA;
    TableParams tp;
    tp.dt = a.dt;
    tp.dt_bias = a.dt_bias;
    tp.A = a.A;
    tp.D = a.D;
    tp.out = tables;
    tp.cost = costs;
    tp.decay = decay;
    tp.L = d.seqlen;
    tp.H = static_cast<int>(d.nheads);
    tp.nblk = static_cast<int>(pl.nblk);
    tp.hpc = d.headdim == 2 * kP ? 1 : kHG;
    tp.chains_per_b = static_cast<int>(d.nheads / tp.hpc);
    tp.dt_min = a.dt_min;
    tp.dt_max = a.dt_max;
    tp.seq = a.seq_idx;
    tp.total = static_cast<int>(pl.total);
    tp.counters = static_cast<uint32_t*>(ws);
    tp.status = a.status_word;
    tp.ncounters = 1 + pl.ncta;
    tp.order = order;
    tp.G = static_cast<int>(d.ngroups);
    tp.sort_pairs = (tp.hpc == kHG && d.nheads <= kSortMaxHeads && d.nheads * (d.nheads / d.ngroups) <= kSortMaxWork)
                        ? 1 : 0;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t tcfg = {};
    // two jobs per warp once one per warp would take more than a wave of CTAs (fewer CTAs rank the heads)
    tp.jobs_per_warp = pl.total > static_cast<long long>(kTableWarps) * kTableCtasPerSm * pl.ncta ? 2 : 1;
    const long long per_cta = static_cast<long long>(kTableWarps) * tp.jobs_per_warp;
    tcfg.gridDim = dim3(static_cast<unsigned>((pl.total + per_cta - 1) / per_cta));
    tcfg.blockDim = dim3(kTableWarps * 32);
    tcfg.stream = a.stream;
    tcfg.attrs = pdl;
    tcfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&tcfg, chain_tables, tp) != cudaSuccess) return SSD_ERR_CUDA;
    // chain_masks and the chain kernel start early as well (programmatic stream
    // serialization) and wait on the device for what they read
    cudaLaunchConfig_t mcfg = {};
    mcfg.gridDim = dim3(static_cast<unsigned>(pl.ntiles));
    mcfg.blockDim = dim3(128);
    mcfg.dynamicSmemBytes = mask_smem<NS>();
    mcfg.stream = a.stream;
    mcfg.attrs = pdl;
    mcfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&mcfg, chain_masks<NS>, tb, tc, masks, static_cast<int>(pl.nblk), static_cast<int>(d.ngroups),
                           a.status_word) != cudaSuccess)
        return SSD_ERR_CUDA;
    uint32_t* ctr = static_cast<uint32_t*>(ws);  // ticket, flags [ncta]
    // with fewer than kBalanceMin jobs per CTA the jobs are split evenly by count
    const bool balance = pl.total >= static_cast<long long>(kBalanceMin) * pl.ncta;
    ChainParams p;
    p.dt = a.dt;
    p.dt_bias = a.dt_bias;
    p.A = a.A;
    p.D = a.D;
    p.init = a.init;
    p.final_state = a.final_state;
    p.x = static_cast<const __nv_bfloat16*>(a.x);
    p.y = static_cast<__nv_bfloat16*>(a.y);
    p.masks = masks;
    p.tables = tables;
    p.ticket = ctr;
    p.flags = ctr + 1;
    p.cost = balance ? costs : nullptr;
    p.job_cost = costs;
    p.decay = decay;
    p.order = order;
    p.warmup = a.chain_warmup;
    p.handoff = handoff;
    p.status = a.status_word;
    p.batch = static_cast<int>(d.batch);
    p.H = static_cast<int>(d.nheads);
    p.G = static_cast<int>(d.ngroups);
    p.nblk = static_cast<int>(pl.nblk);
    p.nchains = static_cast<int>(pl.nchains);
    p.ncta = pl.ncta;
    p.L = d.seqlen;
    p.total = pl.total;
    p.chain_wait_ns = a.wait_limit_ns;
    p.dt_min = a.dt_min;
    p.dt_max = a.dt_max;
    auto* kernel = d.headdim == 2 * kP ? ssd_chain_fused<NS, 2 * kP> : ssd_chain_fused<NS, kP>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Cfg::SMEM_BYTES)) != cudaSuccess)
        return SSD_ERR_CUDA;
    cudaLaunchConfig_t ccfg = {};
    ccfg.gridDim = dim3(static_cast<unsigned>(pl.ncta));
    ccfg.blockDim = dim3(kThreads);
    ccfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    ccfg.stream = a.stream;
    ccfg.attrs = pdl;
    ccfg.numAttrs = 1;
    timing_begin(a.stream);
    if (cudaLaunchKernelEx(&ccfg, kernel, tx, tb, tc, tl, ty, p) != cudaSuccess) return SSD_ERR_CUDA;
    timing_end(a.stream);
    note_launches(3);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

bool chain_supported(const ssd_dims& d, ssd_dtype io, int chunk_len) {
    if (io != SSD_BF16) return false;
    if ((d.headdim != kP && d.headdim != 2 * kP) || (d.dstate != 128 && d.dstate != 256)) return false;
    if (chunk_len != 128 && chunk_len != 256) return false;
    // a chain's two heads share a B/C group (at headdim 128 a chain is one head)
    if (d.headdim == kP && (d.nheads / d.ngroups) % kHG != 0) return false;
    if (d.seqlen >= (1ll << 31) || d.batch >= (1ll << 20) || d.nheads >= (1 << 20)) return false;
    const long long nblk = (d.seqlen + kT - 1) / kT;
    if (nblk * d.batch * d.nheads >= (1ll << 31)) return false;   // job indices are 32-bit
    if (nblk * d.batch * d.ngroups >= (1ll << 31)) return false;  // so are mask tile indices
    return true;
}

size_t chain_workspace_bytes(const ssd_dims& d) {
    int nsm = sm_count();
    if (nsm <= 0) nsm = 1024;  // no device to ask: size for the largest CTA count a device may have
    const ChainPlan pl = plan(d, nsm);
    return chain_ws_bytes(pl);
}

ssd_status chain_forward(const FwdArgs& a, void* ws, size_t ws_bytes) {
    const int nsm = sm_count();
    if (nsm <= 0) return SSD_ERR_CUDA;
    const ChainPlan pl = plan(a.d, nsm);
    if (ws_bytes < chain_ws_bytes(pl)) return SSD_ERR_WORKSPACE;
    for (const void* p : {a.x, static_cast<const void*>(a.B), static_cast<const void*>(a.C),
                          static_cast<const void*>(a.y)})
        if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return SSD_ERR_UNSUPPORTED;
    return a.d.dstate == 256 ? launch_chain<256>(a, ws, pl) : launch_chain<128>(a, ws, pl);
}

}  // namespace ssd
