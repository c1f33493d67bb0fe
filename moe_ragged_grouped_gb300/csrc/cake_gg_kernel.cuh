// cake_gg_kernel.cuh -- persistent, warp-specialised tcgen05 grouped GEMM for sm_103a.
//
// One kernel template serves the three passes of the ragged grouped GEMM
// (flashinfer PR #8258, opening summary: Y = X W^T, dX = G W, dW = G^T X,
// FP32 accumulation, BF16 or FP32 output).  Each CTA owns one SM:
//
//   warp 0      TMA producer: 2-D / 3-D tensor copies into a ring of
//               `stages` shared-memory stages (full / empty mbarriers)
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma.kind::f16, 128 x tile_n
//               x 16 per instruction, FP32 accumulators in two TMEM buffers so
//               the epilogue of one tile overlaps the main loop of the next
//   warps 2..5  epilogue: tcgen05.ld -> registers -> BF16 (round to nearest
//               even, once) or FP32 -> global, masked at expert and tensor
//               edges; the weight gradient's split tiles finish through a
//               per-tile ticket (PR #8258, opening summary, 2nd paragraph: the
//               CTA that arrives last on a tile reads the summed partials and
//               stores the output tile), summing the FP32 partials in split
//               order in deterministic mode or through FP32 atomic adds
//               otherwise.
//
// Operands are staged with a 128-byte swizzle.  K-major tiles (rows of 64
// reduction elements) come from one box of {64, rows}; MN-major tiles come
// from boxes of {64 MN, 64 reduction rows}, 8 KB each, placed 8 KB apart.
//
// Every wait is bounded (timeout_ns, global timer).  On expiry the CTA records
// CAKE_GG_ERR_TIMEOUT in the status word, stops issuing work, waits (bounded)
// for its own copies and MMAs in flight, frees its TMEM and returns.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "cake_gg_ptx.cuh"
#include "cake_gg_sched.h"

namespace cakegg {

constexpr int kThreads = 192;
constexpr int kThreadsRouter = 320;   // + 4 converter warps
constexpr int kThreadsEpi2 = 320;     // forward / data gradient: + a second epilogue warpgroup
constexpr uint32_t kRouterABytes = kTileM * 64 * 4;   // 32 KB: a 128 x 64 FP32 A tile, later its BF16 hi | lo

__host__ __device__ constexpr int threads_for(int kmode)
{
    return kmode == kModeRouter ? kThreadsRouter : kmode == kModeWgrad || kmode == kModeWgradNT ? kThreads : kThreadsEpi2;
}
constexpr int kMaxStages = 8;
constexpr int kMaxCsplit = 8;   // largest cluster split (portable cluster size)
constexpr int kStatusBadOffsets = 7;
constexpr int kStatusTimeout = 8;
constexpr uint32_t kABytes = kTileM * kTileK * 2;  // 16 KB: A tile of one 64-deep k-chunk
constexpr uint32_t kBoxBytes = 64 * 64 * 2;        // one 64 x 64 MN-major box (8 KB)
constexpr size_t kSmemOptInLimit = 232448;        // opt-in dynamic shared memory per CTA (227 KB)
constexpr uint32_t kStagingBytes = 4 * 32 * 128;   // epilogue: 32 rows x 128 B per epilogue warp and buffer

struct KParams {
    const int32_t *offsets;
    void *out;
    int32_t *status;
    uint64_t *tickets;      // per split output tile: (epoch << 32) | arrivals, then slices claimed
    uint64_t spin_ns;       // how long an early split waits for its tile's other partials (0 = never)
    float *partials;
    int64_t M_max;
    int32_t E, N, K;
    int32_t bn;
    int32_t bk;             // reduction elements per stage: 64 * k-chunks per stage
    int32_t stages;
    int32_t kchunk;
    int32_t det;
    int32_t tmem_cols;
    int32_t tma_store;      // epilogue through shared memory + TMA tensor stores
    uint32_t *epoch_word;   // workspace word: the last call's ticket tag (this call uses it + 1, never 0)
    int32_t retire;         // CTAs count their retirement; the last resets the counters and advances the tag
    int32_t stack_a;        // MN-major A through an atom-stacked map: one box per stage
    int32_t stack_b;        // MN-major B likewise (all of this CTA's B atoms in one box)
    int32_t chunk_a;        // K-major A through a {64, rows, K/64} map: one box per stage
    int32_t chunk_b;        // K-major B (forward W) through a {64, N, K/64, E} map
    int32_t pdl;            // launched with programmatic stream serialization
    int32_t staging_bufs;   // epilogue staging buffers per warp (1 or 2)
    int32_t epi_groups;     // forward / data gradient: epilogue warpgroups taking alternate tiles (1 or 2)
    int32_t csplit;         // weight gradient: splits per tile reduced on chip by one cluster (0 = off)
    int32_t debug_flags;
    int32_t prefetch;       // weight gradient: L2 prefetch distance in stages (0 = off)
    int32_t dyn;            // units fetched from a global counter (else a static stride)
    int32_t tail;           // weight gradient: split tail units ...
    int32_t tail_s;         // ... and pieces per tail unit (0 = none)
    int32_t sk;             // weight gradient of one expert: stream-K segment length in k-blocks (0 = off)
    int32_t ntail;          // weight gradient: N-split tail units ...
    int32_t ntq;            // ... and column pieces per tail unit (0 = none)
    int32_t kstagger;       // router: unit t walks its k-blocks from (t * kstagger) mod their count (0 = in order)
    int32_t *sched;         // [0]: next unit, [32]: CTAs retired (zero between calls)
    uint64_t timeout_ns;
};

constexpr int kUQ = 4;      // depth of the queue that passes fetched units to every role

// Control block after the operand ring.
struct __align__(16) Ctrl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t conv[kMaxStages];  // router: the stage's A tile is split into BF16 hi | lo (both CTAs of a pair)
    uint64_t drain;
    uint64_t red_ready;     // cluster split: every split's part of this CTA's slice has arrived
    uint64_t red_consumed;  // cluster split: every peer has read this CTA's partial (pairs: every
                            // owner's ring is free for this tile's parts)
    uint64_t ring_free;     // cluster split of pairs: this CTA's slice is summed, its ring free for copies
    uint64_t uq_full[kUQ];  // unit queue slot written (by the even CTA's producer)
    uint64_t uq_empty[kUQ]; // (even CTA) every role of the cluster has read the slot
    int64_t uq[kUQ];        // unit ids, -1 = no more
    uint32_t tmem_base;
    int32_t abort_flag;
    int32_t bad;
    int32_t last_flag;
    int32_t claim;          // split finish: the slice the epilogue claimed last
    uint32_t epoch;         // this call's ticket tag (read from the workspace at set-up)
    int32_t tail_whole;     // weight gradient: the split tail runs whole (slack placement, decided at set-up)
};

// Walk tables after the control block, sized by the launch's E: off[E+1]
// offsets, order[E] processing position -> expert, pref[E+1] unit prefix in
// processing order, spref[E+1] split prefix by expert id (16-byte aligned).
__host__ __device__ constexpr size_t tables_bytes_for(int E)
{
    return (size_t(4 * E + 3) * 4u + 15u) / 16u * 16u;
}

// A stage holds kps = bk / 64 k-chunks of A (128 rows) and B (bn rows).
// One ring stage: A (128 rows) and this CTA's rows of B (all bn of them, or
// half of them in a 2-SM pair), kps 64-deep k-chunks each.
__host__ __device__ constexpr uint32_t stage_bytes_for(int bn, int kps = 1, int pair = 1, bool router = false)
{
    // router: a 64-deep stage of FP32 A (split in place into BF16 hi | lo) and
    // this CTA's BF16 W rows twice (high, then low parts)
    return router ? kRouterABytes + 2u * uint32_t(bn / pair) * 128u
                  : uint32_t(kps) * (kABytes + uint32_t(bn / pair) * 128u);
}

// Cluster split: the receive buffer of this CTA's slice of a tile's float4
// columns, one copy per split (S x ceil(cols4 / S) <= cols4 + S - 1 columns of
// 128 rows x 16 bytes).  Pairs receive into their operand ring instead (idle
// between a tile's last MMA and the next tile's first copy).
__host__ __device__ constexpr size_t csplit_bytes_for(int bn, int csplit, int pair = 1)
{
    return csplit > 0 && pair == 1 ? size_t(kTileM) * 16u * size_t(bn / 4 + csplit) : 0u;
}

// Cluster split of pairs: float4 columns of a tile's slice owned by one split
// (whole 128-byte output rows per owner: 8 float4 columns for FP32, 16 for BF16)
// and the ring bytes it takes: the receive buffer (the S - 1 peers' parts of
// the slice), then the slice's output staged for TMA stores (per warp, one 4 KB slab of
// 32 rows x 128 bytes per 128-byte row chunk).
// A slice too large for the ring is reduced in `rounds` windows of per / rounds
// columns (per a multiple of rounds row chunks).
__host__ __device__ constexpr int pair_csplit_per(int cols4, int csplit, bool out_f32, int rounds = 1)
{
    return ((cols4 + csplit - 1) / csplit + rounds * (out_f32 ? 8 : 16) - 1) / (rounds * (out_f32 ? 8 : 16)) *
           (rounds * (out_f32 ? 8 : 16));
}
__host__ __device__ constexpr size_t pair_csplit_ring_bytes(int bn, int csplit, bool out_f32, int rounds = 1)
{
    return size_t(csplit - 1) * size_t(pair_csplit_per(bn / 4, csplit, out_f32, rounds) / rounds) * size_t(kTileM) *
               16u +
           4u * size_t(pair_csplit_per(bn / 4, csplit, out_f32, rounds) / rounds / (out_f32 ? 8 : 16)) * 4096u;
}
// Fewest rounds (1, 2 or 4) whose window fits a ring of ring_bytes; 0 if none.
__host__ __device__ constexpr int pair_csplit_rounds(int bn, int csplit, bool out_f32, size_t ring_bytes)
{
    return pair_csplit_ring_bytes(bn, csplit, out_f32, 1) <= ring_bytes   ? 1
           : pair_csplit_ring_bytes(bn, csplit, out_f32, 2) <= ring_bytes ? 2
           : pair_csplit_ring_bytes(bn, csplit, out_f32, 4) <= ring_bytes ? 4
                                                                          : 0;
}

__host__ __device__ constexpr size_t smem_bytes_for(int bn, int stages, int kps, int staging_bufs, int csplit,
                                                    int pair, int E, bool router = false)
{
    return 1024 + size_t(stages) * stage_bytes_for(bn, kps, pair, router) + size_t(staging_bufs) * kStagingBytes +
           csplit_bytes_for(bn, csplit, pair) + sizeof(Ctrl) + tables_bytes_for(E);
}

// Bounded wait on one mbarrier phase, by every lane of the calling warp;
// returns a warp-uniform verdict (false: timed out or another role aborted).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, Ctrl *c,
                                          const KParams &p)
{
    bool ok = mbar_try_wait(bar, parity);
    if (!ok) {
        const uint64_t t0 = global_timer_ns();
        while (true) {
            for (int i = 0; i < 32 && !ok; ++i) ok = mbar_try_wait(bar, parity);
            if (ok) break;
            if (*reinterpret_cast<volatile int32_t *>(&c->abort_flag)) break;
            if (global_timer_ns() - t0 > p.timeout_ns) {
                *reinterpret_cast<volatile int32_t *>(&c->abort_flag) = 1;
                atomicCAS(p.status, 0, kStatusTimeout);
                break;
            }
        }
    }
    return __all_sync(0xffffffffu, ok);
}

// Bounded warp-uniform wait with cluster-scope acquire (barriers that peers
// arrive on remotely).
__device__ __forceinline__ bool cluster_wait(uint32_t bar, uint32_t parity, Ctrl *c, const KParams &p)
{
    bool ok = mbar_try_wait_cluster(bar, parity);
    if (!ok) {
        const uint64_t t0 = global_timer_ns();
        while (true) {
            for (int i = 0; i < 32 && !ok; ++i) ok = mbar_try_wait_cluster(bar, parity);
            if (ok) break;
            if (*reinterpret_cast<volatile int32_t *>(&c->abort_flag)) break;
            if (global_timer_ns() - t0 > p.timeout_ns) {
                *reinterpret_cast<volatile int32_t *>(&c->abort_flag) = 1;
                atomicCAS(p.status, 0, kStatusTimeout);
                break;
            }
        }
    }
    return __all_sync(0xffffffffu, ok);
}

// Same, for a single thread.
__device__ __forceinline__ bool thread_wait(uint32_t bar, uint32_t parity, Ctrl *c,
                                            const KParams &p, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*reinterpret_cast<volatile int32_t *>(&c->abort_flag)) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            *reinterpret_cast<volatile int32_t *>(&c->abort_flag) = 1;
            atomicCAS(p.status, 0, kStatusTimeout);
            return false;
        }
    }
}

// Wait for a phase regardless of the abort flag (used to drain copies / MMAs
// already in flight before the CTA releases its memory).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) return;
    }
}

// Single-thread bounded wait with cluster-scope acquire.
__device__ __forceinline__ bool thread_wait_cluster(uint32_t bar, uint32_t parity, Ctrl *c, const KParams &p)
{
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait_cluster(bar, parity)) return true;
        if (*reinterpret_cast<volatile int32_t *>(&c->abort_flag)) return false;
        if (global_timer_ns() - t0 > p.timeout_ns) {
            *reinterpret_cast<volatile int32_t *>(&c->abort_flag) = 1;
            atomicCAS(p.status, 0, kStatusTimeout);
            return false;
        }
    }
}

// The units a CTA (pair) processes: a static stride over the walk, or, when
// p.dyn, units taken from a global counter in walk order (heaviest first) by
// the even CTA's producer -- greedy list scheduling, so skewed experts
// balance -- and passed to every role of both CTAs through the unit queue.
// Results do not depend on which CTA computes a unit.
struct UnitSeq {
    int64_t t;
    int64_t pos;
};

// A consuming warp (MMA / relay, epilogue) takes the next unit; false = none
// left (or abort: ok = false).
__device__ __forceinline__ bool warp_next_unit(UnitSeq &u, int64_t unit0, int64_t unit_step, int64_t total,
                                               bool leader, uint32_t lead, int lane, Ctrl *c, const KParams &p,
                                               bool &ok)
{
    if (!p.dyn) {
        u.t = u.pos == 0 ? unit0 : u.t + unit_step;
        ++u.pos;
        return u.t < total;
    }
    const int slot = int(u.pos % kUQ);
    const uint32_t par = uint32_t((u.pos / kUQ) & 1);
    const bool w = leader ? warp_wait(smem_u32(&c->uq_full[slot]), par, c, p)
                          : cluster_wait(smem_u32(&c->uq_full[slot]), par, c, p);
    if (!w) {
        ok = false;
        return false;
    }
    u.t = *reinterpret_cast<volatile int64_t *>(&c->uq[slot]);
    __syncwarp();
    if (lane == 0) {
        if (leader) mbar_arrive(smem_u32(&c->uq_empty[slot]));
        else mbar_arrive_remote(map_to_cta(smem_u32(&c->uq_empty[slot]), lead));
    }
    ++u.pos;
    return u.t >= 0;
}

// Ticket of a split output tile: returns how many splits of this call (epoch)
// arrived before this one.  A ticket word left by an earlier call carries
// another epoch and counts as zero, so tickets never need clearing.  At most
// S concurrent updates race, so the CAS loop ends within S tries (bounded at
// 64; on exhaustion the caller is told it is not last and the status word
// records a timeout).
// A claim on a split tile's ticket word once it holds all S arrivals of this
// call: the old count minus S is the next 64-column slice to reduce (>= the
// slice count: none left).  A plain fetch-and-add, so it can be in flight
// while the previous slice is reduced.
__device__ __forceinline__ unsigned long long ticket_claim(uint64_t *t)
{
    return atomicAdd(reinterpret_cast<unsigned long long *>(t), 1ull);
}

__device__ __forceinline__ uint32_t ticket_arrive(uint64_t *t, uint32_t epoch, int32_t *status)
{
    uint64_t cur = *reinterpret_cast<volatile uint64_t *>(t);
    for (int i = 0; i < 64; ++i) {
        const bool same = uint32_t(cur >> 32) == epoch;
        const uint64_t nxt = same ? cur + 1 : ((uint64_t(epoch) << 32) | 1ull);
        const uint64_t prev = atomic_cas_acq_rel_gpu_u64(t, cur, nxt);
        if (prev == cur) return same ? uint32_t(cur & 0xffffffffu) : 0u;
        cur = prev;
    }
    atomicCAS(status, 0, kStatusTimeout);
    return 0xffffffffu;
}

// ---------------------------------------------------------------- epilogue stores

// 32 consecutive columns of one output row (non-transposed), masked at 8-column
// granularity (the row length is a multiple of 8).
template <bool OUT_F32>
__device__ __forceinline__ void store_row32(void *out, int64_t elem_off, int32_t cols_left,
                                            const float (&v)[32])
{
    if (OUT_F32) {
        float *dst = static_cast<float *>(out) + elem_off;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            if (g * 8 < cols_left) {
                float4 *d4 = reinterpret_cast<float4 *>(dst + g * 8);
                d4[0] = make_float4(v[g * 8 + 0], v[g * 8 + 1], v[g * 8 + 2], v[g * 8 + 3]);
                d4[1] = make_float4(v[g * 8 + 4], v[g * 8 + 5], v[g * 8 + 6], v[g * 8 + 7]);
            }
        }
    } else {
        uint16_t *dst = static_cast<uint16_t *>(out) + elem_off;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            if (g * 8 < cols_left) {
                uint4 q;
                q.x = pack_bf16x2(v[g * 8 + 0], v[g * 8 + 1]);
                q.y = pack_bf16x2(v[g * 8 + 2], v[g * 8 + 3]);
                q.z = pack_bf16x2(v[g * 8 + 4], v[g * 8 + 5]);
                q.w = pack_bf16x2(v[g * 8 + 6], v[g * 8 + 7]);
                *reinterpret_cast<uint4 *>(dst + g * 8) = q;
            }
        }
    }
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float x)
{
    return static_cast<uint16_t>(pack_bf16x2(x, 0.0f) & 0xFFFFu);
}

template <bool OUT_F32>
__device__ __forceinline__ void store_scalar(void *out, int64_t idx, float v)
{
    if (OUT_F32) static_cast<float *>(out)[idx] = v;
    else static_cast<uint16_t *>(out)[idx] = f32_to_bf16_rn(v);
}

// Finish of one row of one slice (float4 columns [c4_begin, c4_end)) of a
// split output tile: the FP32 partials p_0 .. p_{nsum-1} (each laid out
// [col/4][row] float4, slot_stride floats apart) are summed in split order
// (s = p_0; s += p_1; ...) and row `lrow` of the slice is written (transposed
// for swapped operands).
// Each batch loads CB float4 columns of SB slots: SB * CB independent
// 16-byte loads in flight per thread.  A lone accumulator (non-deterministic
// splits) is zeroed as it is read, ready for the next call.
template <int CB, int SB, bool OUT_F32, bool TRANSPOSED>
__device__ __forceinline__ void finish_split_row(float *base0, int nsum, int64_t slot_stride, bool zero_after,
                                                 int c4_begin, int c4_end, int lrow, bool row_ok,
                                                 int32_t cols_valid, void *out, int64_t out_base, int64_t ld)
{
    for (int c4 = c4_begin; c4 < c4_end; c4 += CB) {
        float4 acc[CB];
        for (int s0 = 0; s0 < nsum; s0 += SB) {
            float4 b[SB][CB];
#pragma unroll
            for (int u = 0; u < SB; ++u)
#pragma unroll
                for (int j = 0; j < CB; ++j)
                    if (s0 + u < nsum)
                        b[u][j] = __ldcg(reinterpret_cast<const float4 *>(
                            base0 + (s0 + u) * slot_stride + (int64_t(c4 + j) * kTileM + lrow) * 4));
            if (zero_after) {
#pragma unroll
                for (int j = 0; j < CB; ++j)
                    *reinterpret_cast<float4 *>(base0 + (int64_t(c4 + j) * kTileM + lrow) * 4) =
                        make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < SB; ++u) {
                if (s0 + u < nsum) {
#pragma unroll
                    for (int j = 0; j < CB; ++j) {
                        if (s0 + u == 0) {
                            acc[j] = b[u][j];
                        } else {
                            acc[j].x += b[u][j].x;
                            acc[j].y += b[u][j].y;
                            acc[j].z += b[u][j].z;
                            acc[j].w += b[u][j].w;
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < CB; ++j) {
            const int col = (c4 + j) * 4;
            if (row_ok && col < cols_valid) {
                const float vv[4] = {acc[j].x, acc[j].y, acc[j].z, acc[j].w};
                if (TRANSPOSED) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        store_scalar<OUT_F32>(out, out_base + int64_t(col + q4) * ld + lrow, vv[q4]);
                } else if (OUT_F32) {
                    *reinterpret_cast<float4 *>(static_cast<float *>(out) + out_base + int64_t(lrow) * ld + col) =
                        acc[j];
                } else {
                    uint2 pk;
                    pk.x = pack_bf16x2(vv[0], vv[1]);
                    pk.y = pack_bf16x2(vv[2], vv[3]);
                    *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(out) + out_base + int64_t(lrow) * ld + col) =
                        pk;
                }
            }
        }
    }
}

// One warp's 32-row x 128-byte slab of an output tile (this lane's row in w)
// through the warp's staging buffer and a TMA tensor store at (x, y[, z]).
// With two buffers per warp they alternate across every slab the warp ever
// stores (buf persists across tiles), so "all store groups but the newest
// have read their buffers" always covers the buffer written next.
template <int MODE>
__device__ __forceinline__ void stage_and_store(uint8_t *staging, int &buf, int staging_bufs, int q, int lane,
                                                const uint32_t (&w)[32], const CUtensorMap *map, int32_t x,
                                                int32_t y, int32_t z)
{
    uint8_t *stg = staging + (size_t(buf) * 4 + q) * 4096;
    if (lane == 0) {
        // the store that last used this buffer has read it
        if (staging_bufs == 2) bulk_wait_read_but_one();
        else bulk_wait_read_all();
    }
    __syncwarp();
    uint8_t *rowp = stg + lane * 128;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
        *reinterpret_cast<uint4 *>(rowp + ((ch ^ (lane & 7)) << 4)) =
            make_uint4(w[4 * ch], w[4 * ch + 1], w[4 * ch + 2], w[4 * ch + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (MODE == kModeWgrad) tma_store_3d(map, smem_u32(stg), x, y, z);
        else tma_store_2d(map, smem_u32(stg), x, y);
        bulk_commit_group();
    }
    __syncwarp();
    if (staging_bufs == 2) buf ^= 1;
}

// Router: the four K = 16 MMAs of a 64-deep stage with A in tensor memory
// (8 columns per step from a_tmem) and K-major B in shared memory (32 bytes per
// step along the 128-byte swizzled row).
template <int CG>
__device__ __forceinline__ void issue_stage_mmas_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bd0, uint32_t idesc,
                                                    bool first)
{
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
        umma_bf16_ta<CG>(d_tmem, a_tmem + uint32_t(ks) * 8u, bd0 + uint64_t((uint32_t(ks) * 32u) >> 4), idesc,
                         (!first || ks > 0) ? 1u : 0u);
}

// All MMAs of one stage: 4 * KPS k-steps of 16.  Descriptors are built once
// per stage and advanced by adding (byte offset >> 4) to the 14-bit start
// address field (shared-memory addresses stay below 2^18, so no carry).
// MN-major operands step 16 rows (2 KB) down their atoms; K-major operands
// step 32 bytes along the 128-byte row, then to the next 64-deep k-chunk.
template <int KPS, bool A_MN, bool B_MN, int CG>
__device__ __forceinline__ void issue_stage_mmas(uint32_t d_tmem, uint64_t ad0, uint64_t bd0, uint32_t idesc,
                                                 bool first, uint32_t chunk_b)
{
#pragma unroll
    for (int ks = 0; ks < 4 * KPS; ++ks) {
        const uint32_t aoff = A_MN ? uint32_t(ks) * 2048u : uint32_t(ks >> 2) * kABytes + uint32_t(ks & 3) * 32u;
        const uint32_t boff = B_MN ? uint32_t(ks) * 2048u : uint32_t(ks >> 2) * chunk_b + uint32_t(ks & 3) * 32u;
        umma_bf16<CG>(d_tmem, ad0 + uint64_t(aoff >> 4), bd0 + uint64_t(boff >> 4), idesc,
                      (!first || ks > 0) ? 1u : 0u);
    }
}

// Weight gradient: rows [valid, bk) of a stage lie past the expert's end (the
// next expert's rows, or beyond M_max); zero them in every 64-wide atom of
// this CTA's A (2 atoms) and B (natoms - 2 atoms) before the MMAs read the
// stage.  Kept out of line: inlined, it slows the MMA warp's loop on every
// stage although it runs at most once per tile.
static __device__ __noinline__ void zero_stale_rows(uint8_t *ring, uint32_t ring_u32, uint32_t sa, uint32_t sb,
                                                    uint32_t atom_a, uint32_t atom_b, int valid, int bk, int natoms,
                                                    int lane)
{
    // a warp pass covers 4 rows x 8 16-byte chunks of one atom
    const int ch = lane & 7;
    for (int atom = 0; atom < natoms; ++atom) {
        const uint32_t base = atom < 2 ? sa + uint32_t(atom) * atom_a : sb + uint32_t(atom - 2) * atom_b;
        uint8_t *a = ring + (base - ring_u32) + ch * 16;
        for (int row = valid + (lane >> 3); row < bk; row += 4)
            *reinterpret_cast<uint4 *>(a + row * 128) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
}

// A CTA counts itself retired once it will not touch the unit counter again
// (after its last fetch, or at set-up if it takes no units from it); the last
// one of the call leaves the counter at zero for the next call (every CTA's
// fetches are done when it counts itself) and stores this call's ticket tag
// (every CTA read the old one at its set-up, before counting itself).
__device__ __forceinline__ void retire_cta(const KParams &p, uint32_t epoch)
{
    __threadfence();
    if (atomicAdd(p.sched + 32, 1) == int32_t(gridDim.x) - 1) {
        atomicExch(p.sched, 0);
        atomicExch(reinterpret_cast<unsigned int *>(p.epoch_word), epoch);
        atomicExch(p.sched + 32, 0);
    }
}

// ---------------------------------------------------------------- kernel

template <int KMODE, bool SWAP, bool OUT_F32, int PAIR>
__global__ void __launch_bounds__(threads_for(KMODE), 1)
    cake_gg_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                   const __grid_constant__ CUtensorMap mapOut, const KParams p)
{
    // the router is the forward pass (walk, epilogue) with FP32 A tiles split by converter warps
    constexpr bool RT = KMODE == kModeRouter;
    constexpr bool NT = KMODE == kModeWgradNT;   // N-split tail pieces
    constexpr int MODE = RT ? kModeFwd : NT ? kModeWgrad : KMODE;
    constexpr bool A_MN = (MODE == kModeWgrad);
    constexpr bool B_MN = (MODE != kModeFwd);

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t ring_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t *ring = smem_raw + (ring_u32 - raw_u32);
    const int kps = p.bk / kTileK;                 // k-chunks per stage
    const uint32_t stage_bytes = stage_bytes_for(p.bn, kps, PAIR, RT);
    const uint32_t a_bytes = RT ? kRouterABytes : uint32_t(kps) * kABytes;
    const uint32_t atom_a = uint32_t(kps) * kBoxBytes;   // MN-major: 64 x bk atom
    const uint32_t atom_b = atom_a;
    const uint32_t chunk_b = uint32_t(p.bn / PAIR) * 128u;  // K-major B: one 64-deep chunk of this CTA's rows
    uint8_t *staging = ring + size_t(p.stages) * stage_bytes;  // 1024-aligned
    float *red_buf = reinterpret_cast<float *>(staging + size_t(p.staging_bufs) * (p.epi_groups == 2 ? 2 : 1) *
                                               kStagingBytes);
    Ctrl *c = reinterpret_cast<Ctrl *>(reinterpret_cast<uint8_t *>(red_buf) + csplit_bytes_for(p.bn, p.csplit, PAIR));
    int32_t *const t_off = reinterpret_cast<int32_t *>(c + 1);
    int32_t *const t_order = t_off + (p.E + 1);
    int32_t *const t_pref = t_order + p.E;
    int32_t *const t_spref = t_pref + (p.E + 1);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int E = p.E;
    // (cluster splits exist only for weight gradients, swapped single CTAs or
    // pairs: the other instantiations compile none of that path)
    const int csplit = MODE == kModeWgrad && (SWAP || PAIR == 2) ? p.csplit : 0;
    Geom g = make_geom(MODE, E, p.N, p.K, p.M_max, p.bn, SWAP ? 1 : 0, p.kchunk, PAIR, p.bk, csplit,
                       MODE == kModeWgrad ? p.tail : 0, MODE == kModeWgrad ? p.tail_s : 0,
                       MODE == kModeWgrad && !SWAP ? p.sk : 0, NT && !SWAP ? p.ntail : 0, NT && !SWAP ? p.ntq : 0);
    // a cluster shares each unit: a pair (2 CTAs) computes m-tiles 2 * unit + h
    // as one 256-row MMA (the even CTA issues it; each CTA holds its A rows and
    // half of the B tile); a cluster split (csplit CTAs, or csplit pairs)
    // computes one tile, split s taking the s-th chunk of its reduction.  A
    // pair is two CTAs whose cluster ranks differ in bit 0.
    const int cl = PAIR * (csplit > 0 ? csplit : 1);
    const int rank = cl > 1 ? int(cluster_ctarank()) : 0;
    const int half = PAIR == 2 ? (rank & 1) : 0;   // this CTA's half of its pair
    const uint32_t lead = uint32_t(rank - half);  // cluster rank of its pair's even CTA
    const int srank = rank / PAIR;                // cluster split: this CTA's split
    const int64_t unit0 = blockIdx.x / cl;
    const int64_t unit_step = gridDim.x / cl;
    const uint16_t pair_mask = uint16_t(0x3u << lead);
    const bool leader = PAIR == 1 || half == 0;     // issues the MMAs (and owns full / tempty)

    // ---- setup, part 1: TMEM, barriers and tensor maps (no global loads) ----
    // runs while the previous kernel in the stream may still be finishing; the
    // offsets are only pulled into L2 (a prefetch returns no value, so it
    // cannot observe them before that kernel's writes)
    if (warp == 0 && lane * 32 <= E) prefetch_l2(p.offsets + lane * 32);
    if (tid == 0) {
        c->abort_flag = 0;
        c->bad = 0;
        tma_prefetch_desc(&mapA);
        tma_prefetch_desc(&mapB);
        if (p.tma_store) tma_prefetch_desc(&mapOut);
    }
    if (warp == 1) {
        tmem_alloc<PAIR>(smem_u32(&c->tmem_base), uint32_t(p.tmem_cols));
        tmem_relinquish<PAIR>();
    }
    if (tid == 64) {
        for (int s = 0; s < p.stages; ++s) {
            // the even CTA of a pair also counts its peer's "stage loaded" relay
            // (router: the relay is the peer converters' "stage split" on conv)
            mbar_init(smem_u32(&c->full[s]), PAIR == 2 && leader && !RT ? 2u : 1u);
            mbar_init(smem_u32(&c->empty[s]), 1);
            if (RT) mbar_init(smem_u32(&c->conv[s]), PAIR == 2 && leader ? 2u : 1u);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&c->tfull[a]), 1);
            mbar_init(smem_u32(&c->tempty[a]), 4u * PAIR);  // both CTAs' epilogue warps
        }
        mbar_init(smem_u32(&c->drain), 1);
        for (int i = 0; i < kUQ; ++i) {
            mbar_init(smem_u32(&c->uq_full[i]), 1);
            // readers of a slot: MMA (or relay) warp, 4 epilogue warps (8 with a
            // second group), the odd CTA's producer in a pair, and the router's 4
            // converter warps
            mbar_init(smem_u32(&c->uq_empty[i]),
                      (PAIR == 2 ? 11u : 5u) + (RT ? 4u * PAIR : 0u) + (p.epi_groups == 2 ? 4u * PAIR : 0u));
        }
        if (csplit > 0) {
            // single CTAs: this CTA's arrival, the peers' bytes as tx; pairs: this
            // CTA's arrival and one release arrival per pushing thread of every peer
            mbar_init(smem_u32(&c->red_ready), PAIR == 2 ? 1u + uint32_t(csplit - 1) * 128u : 1u);
            mbar_init(smem_u32(&c->red_consumed), uint32_t(csplit));
            mbar_init(smem_u32(&c->ring_free), 1u);
        }
        fence_barrier_init();
    }

    // ---- setup, part 2: offsets, validation, walk tables ----
    // the previous kernel's writes are visible from here on; the next kernel may
    // start its own part 1
    grid_dependency_wait();
    grid_launch_dependents();
    // the producer's first unit from the counter: its round trip overlaps the
    // offsets load and the table build (a stream-K walk takes no counter units)
    int32_t first_fetch = 0;
    const bool fetcher = p.dyn && leader && !(MODE == kModeWgrad && g.sk > 0);   // takes units from the counter
    if (tid == 0 && fetcher) first_fetch = atomicAdd(p.sched, 1);
    if (tid == 32 && p.retire) {
        // this call's ticket tag: one past the last call's, which the previous
        // call's last CTA wrote (a call replayed from a CUDA graph advances too)
        uint32_t e = *reinterpret_cast<volatile uint32_t *>(p.epoch_word) + 1u;
        c->epoch = e == 0 ? 1u : e;
    }
    if (E <= 32) {
        // one warp builds every table: lane e holds expert e
        if (warp == 0) {
            const uint32_t full_mask = 0xffffffffu;
            const int e = lane;
            int32_t a = 0, b = 0;
            if (e < E) {
                a = p.offsets[e];
                b = p.offsets[e + 1];
            }
            const bool badl = e < E && ((e == 0 && a != 0) || b < a || (e == E - 1 && int64_t(b) > p.M_max));
            if (__any_sync(full_mask, badl) && lane == 0) c->bad = 1;
            const int32_t rows = b - a > 0 ? b - a : 0;
            const int32_t cnt = e < E ? expert_tiles(g, rows) : 0;
            const int32_t cost = e < E ? expert_cost(g, rows) : 0;
            const int32_t spl = e < E ? expert_splits(g, rows) : 0;
            if (e < E) t_off[e] = a;
            if (e == E - 1) t_off[E] = b;
            int32_t rank = e;
            if (walk_is_sorted(g)) {
                rank = 0;
                for (int j = 0; j < E; ++j) {
                    const int32_t cj = __shfl_sync(full_mask, cost, j);
                    rank += (cj > cost) || (cj == cost && j < e);
                }
            }
            if (e < E) t_order[rank] = e;
            __syncwarp();
            const int32_t op = lane < E ? t_order[lane] : 0;
            int32_t cnt_p = __shfl_sync(full_mask, cnt, op);
            if (lane >= E) cnt_p = 0;
            int32_t inc_t = cnt_p, inc_s = spl;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int32_t ot = __shfl_up_sync(full_mask, inc_t, d);
                const int32_t os = __shfl_up_sync(full_mask, inc_s, d);
                if (lane >= d) {
                    inc_t += ot;
                    inc_s += os;
                }
            }
            if (lane < E) {
                t_pref[lane] = inc_t - cnt_p;
                t_spref[lane] = inc_s - spl;
            }
            if (lane == 31) {
                t_pref[E] = inc_t;
                t_spref[E] = inc_s;
            }
        }
    } else {
        // block-wide build for many experts (temporaries in the ring)
        int32_t *t_cnt = reinterpret_cast<int32_t *>(ring);
        int32_t *t_cost = t_cnt + kMaxE;
        for (int i = tid; i <= E; i += int(blockDim.x)) t_off[i] = p.offsets[i];
        __syncthreads();
        for (int e = tid; e < E; e += int(blockDim.x)) {
            const int32_t a = t_off[e], b = t_off[e + 1];
            if ((e == 0 && a != 0) || b < a || (e == E - 1 && int64_t(b) > p.M_max)) c->bad = 1;
            const int32_t rows = b - a;
            t_cnt[e] = expert_tiles(g, rows < 0 ? 0 : rows);
            t_cost[e] = expert_cost(g, rows < 0 ? 0 : rows);
        }
        __syncthreads();
        if (walk_is_sorted(g)) {
            for (int e = tid; e < E; e += int(blockDim.x)) {
                const int32_t ce = t_cost[e];
                int32_t rank = 0;
                for (int j = 0; j < E; ++j) {
                    const int32_t cj = t_cost[j];
                    rank += (cj > ce) || (cj == ce && j < e);
                }
                t_order[rank] = e;
            }
        } else {
            for (int e = tid; e < E; e += int(blockDim.x)) t_order[e] = e;
        }
        __syncthreads();
        if (warp == 0) {
            // exclusive prefix sums by one warp: tiles in processing order, splits by expert id
            const int per = (E + 31) / 32;
            const int b0 = lane * per;
            int32_t sum_t = 0, sum_s = 0;
            for (int i = b0; i < b0 + per && i < E; ++i) {
                sum_t += t_cnt[t_order[i]];
                sum_s += expert_splits(g, t_off[i + 1] - t_off[i]);
            }
            int32_t inc_t = sum_t, inc_s = sum_s;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int32_t ot = __shfl_up_sync(0xffffffffu, inc_t, d);
                const int32_t os = __shfl_up_sync(0xffffffffu, inc_s, d);
                if (lane >= d) {
                    inc_t += ot;
                    inc_s += os;
                }
            }
            int32_t run_t = inc_t - sum_t, run_s = inc_s - sum_s;
            for (int i = b0; i < b0 + per && i < E; ++i) {
                t_pref[i] = run_t;
                t_spref[i] = run_s;
                run_t += t_cnt[t_order[i]];
                run_s += expert_splits(g, t_off[i + 1] - t_off[i]);
            }
            if (lane == 31) {
                t_pref[E] = inc_t;
                t_spref[E] = inc_s;
            }
        }
    }
    // the set-up temporaries in the ring are overwritten by TMA (async proxy) later
    fence_proxy_async_smem();
    if (MODE == kModeWgrad && g.tail > 0) {
        // slack placement of the split tail, from the walk tables (one thread)
        __syncthreads();
        if (tid == 0) c->tail_whole = !c->bad && tail_fits_whole(g, t_off, t_order, int32_t(kWaveCtas / PAIR)) ? 1 : 0;
    }
    tc_fence_before_sync();
    __syncthreads();
    if (c->bad) {
        // every CTA (and every CTA of a cluster) sees the same offsets and leaves here
        // (counting itself retired, so the counters are zero again after the call)
        if (tid == 0) {
            atomicCAS(p.status, 0, kStatusBadOffsets);
            if (p.retire) retire_cta(p, c->epoch);
        }
        if (warp == 1) {
            tc_fence_after_sync();
            tmem_dealloc<PAIR>(c->tmem_base, uint32_t(p.tmem_cols));
        }
        return;
    }
    // a CTA that takes no units from the counter counts itself retired now (it
    // has read the ticket tag); a fetching one right after its last fetch --
    // both off the kernel's tail
    if (tid == 0 && p.retire && !fetcher) retire_cta(p, c->epoch);
    // peers' barriers must exist before a commit signal or a remote arrive reaches
    // them: warps that reach into peers (all of a pair; the epilogue of a
    // cluster split) wait here, the others only at teardown
    const bool early_wait = PAIR == 2 || warp >= 2;
    if (cl > 1) {
        cluster_arrive_relaxed();
        if (early_wait) cluster_wait_acquire();
    }
    tc_fence_after_sync();

    if (MODE == kModeWgrad && g.tail > 0 && c->tail_whole) g.tail = g.tail_s = 0;
    const int64_t total = walk_length(g, t_pref[E]);
    const uint32_t tmem_base = c->tmem_base;
    const uint32_t acc_stride = uint32_t(p.tmem_cols) / 2;
    // a 512-wide tile fills TMEM: one accumulator, released before the next unit;
    // the router keeps one accumulator (columns 0..255) and the split A tiles of
    // its stages in the columns after it (64 per stage: high, then low parts)
    const int nacc = (p.bn > 256 || RT) ? 1 : 2;

    if (warp == 0) {
        // ======================= TMA producer =======================
        if (lane == 0) {
            const uint32_t tx = stage_bytes;
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            UnitSeq us{0, 0};
            int32_t nxt = 0;
            // stream-K: the leader walks its own virtual pairs (unit0, unit0 + unit_step, ...)
            // and their pieces in order; no counter
            const bool skw = MODE == kModeWgrad && g.sk > 0;
            int32_t sk_K = 0, sk_pm = 1, sk_nv = 0, sk_v = int32_t(unit0), sk_pc = 0;
            if (skw) {
                sk_K = sk_kb(g, t_off[1] - t_off[0]);
                sk_pm = sk_pmax(g, sk_K);
                sk_nv = sk_virtual(g, sk_K);
            }
            if (p.dyn && leader && !skw) nxt = first_fetch;
            while (ok) {
                int64_t t;
                if (!p.dyn) {
                    t = us.pos == 0 ? unit0 : us.t + unit_step;
                    us.t = t;
                    ++us.pos;
                    if (t >= total) break;
                    // cluster split of pairs: the previous tile's parts were received
                    // in this ring; its copies wait until that slice is summed
                    if (PAIR == 2 && csplit > 0 && us.pos > 1 &&
                        !thread_wait(smem_u32(&c->ring_free), uint32_t((us.pos - 2) & 1), c, p, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                } else if (leader) {
                    // fetch: publish the unit to every role of the cluster
                    const int slot = int(us.pos % kUQ);
                    if (us.pos >= kUQ && !thread_wait_cluster(smem_u32(&c->uq_empty[slot]),
                                                              uint32_t(((us.pos / kUQ) - 1) & 1), c, p)) {
                        ok = false;
                        break;
                    }
                    if (skw) {
                        t = -1;
                        while (sk_v < sk_nv) {
                            if (sk_pc < sk_pieces(g, sk_K, sk_v)) {
                                t = int64_t(sk_v) * sk_pm + sk_pc++;
                                break;
                            }
                            sk_v += int32_t(unit_step);
                            sk_pc = 0;
                        }
                    } else {
                        t = int64_t(nxt) < total ? int64_t(nxt) : -1;
                    }
                    c->uq[slot] = t;
                    mbar_arrive(smem_u32(&c->uq_full[slot]));
                    // the odd CTA's slot: data and signal in one asynchronous store
                    // (that CTA armed its barrier for these 8 bytes)
                    if (PAIR == 2)
                        st_async_b64(map_to_cta(smem_u32(&c->uq[slot]), lead + 1u), t,
                                     map_to_cta(smem_u32(&c->uq_full[slot]), lead + 1u));
                    ++us.pos;
                    if (t < 0) break;
                } else {
                    // the odd CTA's producer reads the queue like every other role; it
                    // also arms each slot's barrier for the next 8-byte delivery (the
                    // even CTA writes a slot again only after every reader released it)
                    const int slot = int(us.pos % kUQ);
                    if (us.pos == 0)
                        for (int i = 0; i < kUQ; ++i) mbar_arrive_expect_tx(smem_u32(&c->uq_full[i]), 8u);
                    if (!thread_wait_cluster(smem_u32(&c->uq_full[slot]), uint32_t((us.pos / kUQ) & 1), c, p)) {
                        ok = false;
                        break;
                    }
                    t = *reinterpret_cast<volatile int64_t *>(&c->uq[slot]);
                    if (t >= 0) mbar_arrive_expect_tx(smem_u32(&c->uq_full[slot]), 8u);
                    mbar_arrive_remote(map_to_cta(smem_u32(&c->uq_empty[slot]), lead));
                    ++us.pos;
                    if (t < 0) break;
                }
                const Tile ti = decode_tile(g, t, t_off, t_order, t_pref, t_spref, rank);
                // the next unit is fetched while this one's last stages go out: early
                // enough to hide the atomic, late enough that every CTA of the grid
                // has taken its first unit (fetching at once would let the first
                // pairs to start hold two units while late ones find none)
                const int32_t fetch_kb = ti.kb1 - (p.stages + 1) > ti.kb0 ? ti.kb1 - (p.stages + 1) : ti.kb0;
                bool fetched = !(p.dyn && leader) || skw;
                // (the router staggers each unit's k order: with one output-column
                // tile every pair reads the same weight slices, and in lock step they
                // would all read the same lines at once.  The unit's rotation is
                // taken once here: a 64-bit remainder per stage sat between each
                // stage's wait and its copies, on the one thread that issues them,
                // and cost the router 6 %.)
                const int32_t nk = ti.kb1 - ti.kb0;
                const int32_t krot = RT && p.kstagger > 0 && nk > 0 ? int32_t((t * p.kstagger) % nk) : 0;
                for (int kb = ti.kb0; kb < ti.kb1; ++kb) {
                    if (!fetched && kb == fetch_kb) {
                        nxt = atomicAdd(p.sched, 1);  // in flight while the copies go out
                        fetched = true;
                    }
                    if (!thread_wait(smem_u32(&c->empty[stage]), phase ^ 1u, c, p, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&c->full[stage]);
                    const uint32_t sa = ring_u32 + uint32_t(stage) * stage_bytes;
                    const uint32_t sb = sa + a_bytes;
                    // (an N-split tail piece of a 512-wide tile loads one B box: the
                    // map's 256 / 64 / PAIR atoms from its first one)
                    mbar_arrive_expect_tx(fb, NT && ti.cw < p.bn
                                                  ? a_bytes + uint32_t(256 / 64 / PAIR) * atom_b
                                                  : tx);
                    // test hook: the walk's first unit (whichever CTA takes it) loses its
                    // first copy on the even / single CTA
                    const bool drop = (p.debug_flags & 1) && t == 0 && kb == ti.kb0 && rank == 0;
                    if (!drop) {
                        // B atoms this CTA loads: all of them, or its half of a pair's
                        const int nb = p.bn / 64;
                        const int jb0 = PAIR == 2 ? half * nb / 2 : 0;
                        const int jb1 = PAIR == 2 ? (half + 1) * nb / 2 : nb;
                        int32_t kbr = kb;
                        if (RT) {
                            kbr = kb + krot;
                            if (kbr >= ti.kb1) kbr -= nk;
                        }
                        const int32_t k0 = kbr * p.bk;      // first reduction element of the stage
                        if (MODE == kModeWgrad) {
                            const int32_t r = ti.row0 + k0;
                            // both operands stream once per unit from rows far apart in
                            // time across the grid: pull the stage `prefetch` ahead into
                            // L2 so that its real load hits
                            if (p.prefetch > 0 && kb + p.prefetch < ti.kb1 && p.stack_a && p.stack_b) {
                                const int32_t rp = r + p.prefetch * p.bk;
                                tma_prefetch_l2_3d(&mapA, 0, rp, ti.mt * 2);
                                tma_prefetch_l2_3d(&mapB, 0, rp, ti.nt * nb + jb0);
                            }
                            // A: 128 MN x bk rows as two 64-wide atoms
                            if (p.stack_a) {
                                tma_load_3d(sa, &mapA, fb, 0, r, ti.mt * 2);
                            } else {
                                tma_load_2d(sa, &mapA, fb, ti.mt * kTileM, r);
                                tma_load_2d(sa + atom_a, &mapA, fb, ti.mt * kTileM + 64, r);
                            }
                            if (NT && p.stack_b && p.bn > 256 && ti.cw < p.bn) {
                                // an N-split tail piece of a 512-wide tile: one box from
                                // this CTA's first atom of the piece (cw / PAIR columns,
                                // whole 64-wide atoms); the MMA reads cw / PAIR columns of
                                // it, the rest of the box is the next columns (or the
                                // zero fill past K)
                                const int pa = ti.cw / 64 / PAIR;
                                tma_load_3d(sb, &mapB, fb, 0, r, ti.nt * nb + ti.c0 / 64 + half * pa);
                            } else if (p.stack_b && p.bn > 256) {
                                // a 512-wide tile: this CTA's half of each 256-column MMA tile
                                const int hb = 256 / 64 / PAIR;   // atoms per half per CTA
                                tma_load_3d(sb, &mapB, fb, 0, r, ti.nt * nb + half * hb);
                                tma_load_3d(sb + uint32_t(hb) * atom_b, &mapB, fb, 0, r, ti.nt * nb + 4 + half * hb);
                            } else if (p.stack_b) {
                                tma_load_3d(sb, &mapB, fb, 0, r, ti.nt * nb + jb0);
                            } else {
                                for (int j = jb0; j < jb1; ++j)
                                    tma_load_2d(sb + (j - jb0) * atom_b, &mapB, fb, ti.nt * p.bn + 64 * j, r);
                            }
                        } else if (RT) {
                            // router: the FP32 X tile as two 32-column boxes (128-byte rows,
                            // 128-byte swizzle; converted in place to BF16 hi | lo), then this
                            // CTA's rows of W's BF16 high and low parts (W' = [w_hi | w_lo])
                            tma_load_2d(sa, &mapA, fb, k0, ti.row0);
                            tma_load_2d(sa + kRouterABytes / 2, &mapA, fb, k0 + 32, ti.row0);
                            // the ring is shallow (64 KB stages) and each stage waits for its
                            // split as well: pull X `prefetch` stages ahead into L2
                            if (p.prefetch > 0 && kb + p.prefetch < ti.kb1) {
                                tma_prefetch_l2_2d(&mapA, k0 + p.prefetch * 64, ti.row0);
                                tma_prefetch_l2_2d(&mapA, k0 + p.prefetch * 64 + 32, ti.row0);
                            }
                            const int32_t wrow = ti.nt * p.bn + half * (p.bn / PAIR);
                            tma_load_3d(sb, &mapB, fb, k0, wrow, 0);
                            tma_load_3d(sb + uint32_t(p.bn / PAIR) * 128u, &mapB, fb, p.K + k0, wrow, 0);
                        } else {
                            // K-major A (X or G): all k-chunks of the stage in one box when chunked
                            if (p.chunk_a) tma_load_3d(sa, &mapA, fb, 0, ti.row0, kb * kps);
                            else tma_load_2d(sa, &mapA, fb, k0, ti.row0);
                            if (MODE == kModeFwd && p.bn > 256) {
                                // a 512-wide tile: this CTA's half of each 256-row W block
                                // (K-major: 256 / PAIR rows of 128 bytes per block)
                                const int32_t wrow = ti.nt * p.bn + half * (256 / PAIR);
                                tma_load_3d(sb, &mapB, fb, k0, wrow, ti.e);
                                tma_load_3d(sb + uint32_t(256 / PAIR) * 128u, &mapB, fb, k0, wrow + 256, ti.e);
                            } else if (MODE == kModeFwd) {
                                // this CTA's rows of the W tile: all bn, or its half of a pair's
                                const int32_t wrow = ti.nt * p.bn + half * (p.bn / PAIR);
                                if (p.chunk_b)
                                    tma_load_4d(sb, &mapB, fb, 0, wrow, kb * kps, ti.e);
                                else
                                    tma_load_3d(sb, &mapB, fb, k0, wrow, ti.e);
                            } else if (p.stack_b && p.bn > 256) {
                                // a 512-wide tile: this CTA's half of each 256-column MMA tile
                                const int hb = 256 / 64 / PAIR;
                                tma_load_4d(sb, &mapB, fb, 0, k0, ti.nt * nb + half * hb, ti.e);
                                tma_load_4d(sb + uint32_t(hb) * atom_b, &mapB, fb, 0, k0, ti.nt * nb + 4 + half * hb,
                                            ti.e);
                            } else if (p.stack_b) {
                                // W as {64, N, K/64, E}: this CTA's atoms of one bk-row block in one box
                                tma_load_4d(sb, &mapB, fb, 0, k0, ti.nt * nb + jb0, ti.e);
                            } else {
                                for (int j = jb0; j < jb1; ++j)
                                    tma_load_3d(sb + (j - jb0) * atom_b, &mapB, fb, ti.nt * p.bn + 64 * j, k0, ti.e);
                            }
                        }
                    }
                    ++issued;
                    if (++stage == p.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                // a unit without k-blocks (an empty expert's zero tile) fetches here
                if (!fetched && ok) nxt = atomicAdd(p.sched, 1);
            }
            // the counter's last use by this CTA is behind it
            if (fetcher && p.retire) retire_cta(p, c->epoch);
            if (!ok) {
                // drain: the most recent issue into each stage must land before exit
                const int64_t n = issued < p.stages ? issued : p.stages;
                for (int64_t i = 0; i < n; ++i) {
                    const int64_t q = issued - 1 - i;
                    drain_wait(smem_u32(&c->full[q % p.stages]), uint32_t((q / p.stages) & 1),
                               20000000ull);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ======================= MMA issuer =======================
        // (the odd CTA of a pair issues none: it zeroes its stale rows of each
        // loaded stage and relays "stage loaded" to the even CTA's full barrier)
        // (a 512-wide tile is two MMAs of N = 256 per k-step, into TMEM columns 0 and 256)
        const uint32_t idesc = idesc_bf16_f32(kTileM * PAIR, uint32_t(p.bn > 256 ? 256 : p.bn), A_MN, B_MN);
        // (an N-split tail piece is one MMA of its width per k-step)
        const uint32_t idesc_piece =
            NT ? idesc_bf16_f32(kTileM * PAIR, uint32_t(g.ntq > 1 ? p.bn / g.ntq : p.bn), A_MN, B_MN) : idesc;
        int stage = 0;
        uint32_t phase = 0;
        int it = 0;
        bool ok = true;
        bool any_mma = false;
        for (UnitSeq us{0, 0}; ok && warp_next_unit(us, unit0, unit_step, total, leader, lead, lane, c, p, ok); ++it) {
            const int64_t t = us.t;
            const Tile ti = decode_tile(g, t, t_off, t_order, t_pref, t_spref, rank);
            const int acc = nacc == 2 ? (it & 1) : 0;
            const uint32_t acc_phase = nacc == 2 ? (uint32_t(it >> 1) & 1u) : (uint32_t(it) & 1u);
            if (leader) {
                // every epilogue warp (of both CTAs of a pair) released this buffer
                if (!warp_wait(smem_u32(&c->tempty[acc]), acc_phase ^ 1u, c, p)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
            }
            const uint32_t d_tmem = tmem_base + uint32_t(acc) * acc_stride;
            // weight gradient: the one k-block of this unit whose stage reaches past
            // the expert's end (none when the expert's rows are a multiple of bk)
            int zero_kb = -1, zero_valid = 0;
            if (MODE == kModeWgrad && ti.kb1 > ti.kb0) {
                const int32_t v = ti.row_end - (ti.row0 + (ti.kb1 - 1) * p.bk);
                if (v < p.bk) {
                    zero_kb = ti.kb1 - 1;
                    zero_valid = v;
                }
            }
            for (int kb = ti.kb0; kb < ti.kb1; ++kb) {
                // (the even CTA's full barrier also counts the peer's relay; the
                // router's MMA waits instead for both CTAs' converters on conv,
                // whose waits cover the copies, and the odd CTA's warp has nothing
                // to relay)
                if (RT) {
                    if (leader && !(PAIR == 2 ? cluster_wait(smem_u32(&c->conv[stage]), phase, c, p)
                                              : warp_wait(smem_u32(&c->conv[stage]), phase, c, p))) {
                        ok = false;
                        break;
                    }
                } else if (!warp_wait(smem_u32(&c->full[stage]), phase, c, p)) {
                    ok = false;
                    break;
                }
                const uint32_t sa = ring_u32 + uint32_t(stage) * stage_bytes;
                const uint32_t sb = sa + a_bytes;
                if (MODE == kModeWgrad && kb == zero_kb)
                    zero_stale_rows(ring, ring_u32, sa, sb, atom_a, atom_b, zero_valid, p.bk,
                                    2 + (NT ? ti.cw : p.bn) / 64 / PAIR, lane);
                __syncwarp();
                if (leader) {
                    if (lane == 0) {
                        tc_fence_after_sync();
                        const uint64_t ad0 = A_MN ? smem_desc_sw128(sa, atom_a, 1024) : smem_desc_sw128(sa, 16, 1024);
                        const uint64_t bd0 = B_MN ? smem_desc_sw128(sb, atom_b, 1024) : smem_desc_sw128(sb, 16, 1024);
                        const bool first = kb == ti.kb0;
                        if (RT) {
                            // x_hi w_hi + x_hi w_lo + x_lo w_hi into one accumulator; the
                            // split A tile of this stage is in TMEM (high parts, then low)
                            const uint32_t a_hi = tmem_base + 256u + uint32_t(stage) * 64u;
                            const uint64_t bl = smem_desc_sw128(sb + uint32_t(p.bn / PAIR) * 128u, 16, 1024);
                            issue_stage_mmas_ta<PAIR>(d_tmem, a_hi, bd0, idesc, first);
                            issue_stage_mmas_ta<PAIR>(d_tmem, a_hi, bl, idesc, false);
                            issue_stage_mmas_ta<PAIR>(d_tmem, a_hi + 32u, bd0, idesc, false);
                        } else if (NT && ti.cw < p.bn) {
                            issue_stage_mmas<1, A_MN, B_MN, PAIR>(d_tmem, ad0, bd0, idesc_piece, first, chunk_b);
                        } else if (p.bn > 256) {
                            // this CTA's halves of the two 256-column B tiles sit 2 * (128 / PAIR / 64) atoms apart
                            const uint32_t half = uint32_t(256 / 64 / PAIR) * atom_b;
                            const uint64_t bd1 =
                                B_MN ? smem_desc_sw128(sb + half, atom_b, 1024) : smem_desc_sw128(sb + half, 16, 1024);
                            issue_stage_mmas<1, A_MN, B_MN, PAIR>(d_tmem, ad0, bd0, idesc, first, chunk_b);
                            issue_stage_mmas<1, A_MN, B_MN, PAIR>(d_tmem + 256u, ad0, bd1, idesc, first, chunk_b);
                        } else if (kps == 1)
                            issue_stage_mmas<1, A_MN, B_MN, PAIR>(d_tmem, ad0, bd0, idesc, first, chunk_b);
                        else if (kps == 2) issue_stage_mmas<2, A_MN, B_MN, PAIR>(d_tmem, ad0, bd0, idesc, first, chunk_b);
                        else issue_stage_mmas<4, A_MN, B_MN, PAIR>(d_tmem, ad0, bd0, idesc, first, chunk_b);
                        // the stage is free again in both CTAs once these MMAs complete
                        if (PAIR == 2) umma_commit_mc<2>(smem_u32(&c->empty[stage]), pair_mask);
                        else umma_commit<1>(smem_u32(&c->empty[stage]));
                    }
                    any_mma = true;
                } else if (lane == 0 && !RT) {
                    mbar_arrive_remote(map_to_cta(smem_u32(&c->full[stage]), lead));
                }
                __syncwarp();
                if (++stage == p.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            if (leader && lane == 0) {
                if (PAIR == 2) umma_commit_mc<2>(smem_u32(&c->tfull[acc]), pair_mask);
                else umma_commit<1>(smem_u32(&c->tfull[acc]));
            }
            __syncwarp();
        }
        if (!ok && any_mma) {
            if (lane == 0) {
                umma_commit<PAIR>(smem_u32(&c->drain));
                drain_wait(smem_u32(&c->drain), 0, 20000000ull);
            }
            __syncwarp();
        }
    } else if (!RT || warp < 6) {
        // ======================= epilogue (warps 2..5; 6..9) =======================
        // (forward / data gradient with a short reduction: a second warpgroup,
        // warps 6..9, takes every other tile -- the odd accumulator -- so two
        // warps per SM sub-partition overlap the latency of the stores)
        const int q = warp & 3;            // TMEM lane quarter this warp may access
        const int lrow = q * 32 + lane;    // tile row held by this thread
        const int eg = (warp - 2) >> 2;    // epilogue group
        const int ngroups = p.epi_groups == 2 && nacc == 2 ? 2 : 1;
        const uint32_t ebar = eg == 0 ? 1u : 3u;   // the group's named barrier
        const int etid = (tid - 64) & 127; // 0..127 within the group
        // cluster split of pairs: rounds of the reduction (a slice wider than the ring holds)
        const int cs_rounds =
            PAIR == 2 && csplit > 0 ? pair_csplit_rounds(p.bn, csplit, OUT_F32, size_t(p.stages) * stage_bytes) : 1;
        uint8_t *const stg_base = staging + size_t(eg) * p.staging_bufs * kStagingBytes;
        int it = 0;
        int cs_it = 0;                     // cluster-split tiles reduced so far
        int stg_buf = 0;                   // staging buffer this warp writes next
        bool qok = true;
        // cluster split: the bytes of this CTA's slice that its peers push for
        // the current tile, whether that tile's receive phase is still open (the
        // peers may push into it) and whether this CTA has armed it
        uint32_t cs_expect = 0;
        bool cs_open = false, cs_armed = false;
        for (UnitSeq us{0, 0}; warp_next_unit(us, unit0, unit_step, total, leader, lead, lane, c, p, qok); ++it) {
            if (it % ngroups != eg) continue;   // the other group's tile
            const int64_t t = us.t;
            const Tile ti = decode_tile(g, t, t_off, t_order, t_pref, t_spref, rank);
            const int acc = nacc == 2 ? (it & 1) : 0;
            const uint32_t acc_phase = nacc == 2 ? (uint32_t(it >> 1) & 1u) : (uint32_t(it) & 1u);
            const bool empty_tile = ti.kb1 <= ti.kb0;
            const int32_t tcw = NT ? ti.cw : p.bn;   // columns of the tile this unit computes
            const int32_t tc0 = NT ? ti.c0 : 0;      // ... from this one
            const bool split = (MODE == kModeWgrad) && ti.S > 1 && ti.valid;
            const uint32_t t_row = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(acc) * acc_stride;

            // output geometry of this tile
            int64_t out_base = 0;   // element offset of tile (row 0, col 0)
            int64_t ld = 0;         // row stride (elements) of the output
            int32_t rows_valid = 0; // tile rows that exist
            int32_t cols_valid = 0; // tile columns that exist
            if (MODE == kModeFwd) {
                ld = p.N;
                out_base = int64_t(ti.row0) * ld + int64_t(ti.nt) * p.bn;
                rows_valid = ti.row_end - ti.row0;
                cols_valid = p.N - ti.nt * p.bn;
            } else if (MODE == kModeDgrad) {
                ld = p.K;
                out_base = int64_t(ti.row0) * ld + int64_t(ti.nt) * p.bn;
                rows_valid = ti.row_end - ti.row0;
                cols_valid = p.K - ti.nt * p.bn;
            } else if (!SWAP) {
                // (an N-split tail piece: columns [c0, c0 + cw) of the tile)
                ld = p.K;
                out_base = int64_t(ti.e) * p.N * p.K + int64_t(ti.mt) * kTileM * ld + int64_t(ti.nt) * p.bn + tc0;
                rows_valid = p.N - ti.mt * kTileM;
                cols_valid = p.K - (ti.nt * p.bn + tc0);
            } else {
                // C[m = k, n = n] -> dW[e, n, k]: transposed store
                ld = p.K;
                out_base = int64_t(ti.e) * p.N * p.K + int64_t(ti.nt) * p.bn * ld + int64_t(ti.mt) * kTileM;
                rows_valid = p.K - ti.mt * kTileM;
                cols_valid = p.N - ti.nt * p.bn;
            }
            if (cols_valid > tcw) cols_valid = tcw;
            const bool row_ok = lrow < rows_valid;
            // cluster split: this CTA's float4 columns [q0, q1) of the tile's nq
            // (pairs: whole 128-byte output rows per owner, stored by TMA)
            const int nq = (cols_valid > 0 ? cols_valid : 0) / 4;
            const int per_c = csplit > 0
                                  ? (PAIR == 2 ? pair_csplit_per(nq, csplit, OUT_F32, cs_rounds) : (nq + csplit - 1) / csplit)
                                  : 1;
            const int per = per_c > 0 ? per_c : 1;   // (>= 1: also keeps pruned code free of a zero divisor)
            const int q0 = srank * per;
            const int q1 = q0 + per < nq ? q0 + per : nq;
            if (csplit > 0) {
                cs_expect = uint32_t(csplit - 1) * uint32_t(q1 > q0 ? q1 - q0 : 0) * kTileM * 16u;
                cs_open = true;
                cs_armed = false;
            }

            // (in a pair the even CTA's MMA commit arrives on both CTAs' tfull)
            bool ok = warp_wait(smem_u32(&c->tfull[acc]), acc_phase, c, p);
            ok = named_bar_and(ebar, 128, ok);
            if (!ok) break;
            tc_fence_after_sync();

            if (csplit > 0) {
                // ---- cluster split: partial slices pushed to their owners, summed there ----
                // Split s of the cluster owns float4 columns [s per, (s + 1) per) of the
                // tile (in a pair, of its half's 128 rows); the owner sums every
                // split's part of its slice in split order and stores it.
                // Single CTAs: every CTA pushes its partial's part of each slice into
                // the owner's receive buffer rec[s][q][row] (s = the pushing CTA's
                // split; the owner writes its own part too) with st.async, counted in
                // bytes on the owner's red_ready; before pushing a tile's slices a CTA
                // waits until every owner has summed the previous tile's
                // (red_consumed).
                // Pairs receive into their operand ring: an owner arms its receive
                // phase and signals red_consumed once its pair's MMAs of the tile
                // are complete (this CTA's tfull), pushers wait for every owner's
                // signal, and the owner's producer copies the next tile into the ring
                // only after the slice is summed (ring_free).
                constexpr bool kRing = PAIR == 2;
                uint8_t *rec = kRing ? ring : reinterpret_cast<uint8_t *>(red_buf);
                const uint32_t rec_u32 = smem_u32(rec);
                if (kRing) {
                    // R rounds, round r taking columns [o per + r pr, o per + (r + 1) pr)
                    // of every owner o's slice (pr = per / R): the receive buffer and the
                    // staged output are one window's
                    const int pr = per / (cs_rounds > 0 ? cs_rounds : 1);
                    bool cs_ok = true;
                    for (int rd = 0; rd < cs_rounds; ++rd) {
                        if (rd > 0) {
                            // the previous window is summed and its slabs' stores have read
                            // them: this CTA's window is free again
                            if (lane == 0) bulk_wait_read_all();
                            __syncwarp();
                            fence_proxy_async_smem();
                            named_bar_sync(ebar, 128);
                            cs_open = true;
                        }
                        if (etid == 0) {
                            mbar_arrive(smem_u32(&c->red_ready));
                            for (int j = 0; j < csplit; ++j)
                                mbar_arrive_cluster(map_to_cta(smem_u32(&c->red_consumed), uint32_t(j * PAIR + half)));
                        }
                        cs_armed = true;
                        bool okc = cluster_wait(smem_u32(&c->red_consumed), uint32_t(cs_it & 1), c, p);
                        if (!named_bar_and(ebar, 128, okc)) {
                            cs_ok = false;
                            break;
                        }
                        // Pairs: each owner's window of the other splits' partials goes out
                        // straight from TMEM (whole 32-column chunks: pr is a multiple of 8)
                        // as plain stores into the owner's ring, rec[s'][q - q_window][row]
                        // with s' the pusher's split among the owner's S - 1 peers; the
                        // owner's own part stays in TMEM until its sum.
                        for (int o = 0; o < csplit; ++o) {
                            if (o == srank) continue;
                            const int qa = o * per + rd * pr;
                            const int qb = qa + pr < nq ? qa + pr : nq;
                            const int slot = srank < o ? srank : srank - 1;
                            const uint32_t rbase = map_to_cta(
                                rec_u32 + uint32_t((slot * pr * kTileM + lrow) * 16), uint32_t(o * PAIR + half));
                            for (int qc = qa; qc < qb; qc += 16) {   // two 32-column chunks per TMEM wait
                                uint32_t r0[32], r1[32];
                                const bool two = qc + 8 < qb;
                                if (empty_tile) {
#pragma unroll
                                    for (int j = 0; j < 32; ++j) r0[j] = r1[j] = 0u;
                                } else {
                                    tmem_ld_32x32b_x32(t_row + uint32_t(4 * qc), r0);
                                    if (two) tmem_ld_32x32b_x32(t_row + uint32_t(4 * qc + 32), r1);
                                    tmem_ld_wait();
                                }
#pragma unroll
                                for (int j4 = 0; j4 < 16; ++j4) {
                                    const uint32_t *rr = j4 < 8 ? r0 : r1;
                                    const int jj = j4 & 7;
                                    if (qc + j4 < qb)
                                        st_cluster_v4(rbase + uint32_t((qc + j4 - qa) * kTileM * 16),
                                                      make_float4(__uint_as_float(rr[4 * jj]),
                                                                  __uint_as_float(rr[4 * jj + 1]),
                                                                  __uint_as_float(rr[4 * jj + 2]),
                                                                  __uint_as_float(rr[4 * jj + 3])));
                                }
                            }
                        }
                        // plain stores, made visible by one release arrival per thread on
                        // every other owner (fewer barrier updates than a byte count per store)
                        for (int j = 0; j < csplit; ++j)
                            if (j != srank)
                                mbar_arrive_cluster(map_to_cta(smem_u32(&c->red_ready), uint32_t(j * PAIR + half)));
                        bool okr = cluster_wait(smem_u32(&c->red_ready), uint32_t(cs_it & 1), c, p);
                        if (!named_bar_and(ebar, 128, okr)) {
                            cs_ok = false;
                            break;
                        }
                        cs_open = false;   // every peer's part of the window has landed
                        ++cs_it;
                        // My window, summed over the splits in split order (s = 0, 1, ...,
                        // S - 1; this CTA's own part from TMEM), staged per warp in the ring
                        // after the receive buffer as 4 KB slabs (32 rows x one 128-byte
                        // output row chunk) whose TMA stores go out back to back.
                        constexpr int CW = OUT_F32 ? 32 : 64;   // columns per 128-byte output row
                        constexpr int C4 = CW / 4;
                        const int w0 = q0 + rd * pr;
                        const int w1 = w0 + pr < q1 ? w0 + pr : q1;
                        const uint32_t ostg = rec_u32 + uint32_t(csplit - 1) * uint32_t(pr) * kTileM * 16u +
                                              uint32_t(q) * uint32_t(pr / C4) * 4096u;
                        const bool stage_out = p.tma_store && ti.valid && q * 32 < rows_valid;
                        for (int qc = w0; qc < w1; qc += C4) {
                            // this CTA's own part of the row chunk, from TMEM
                            uint32_t own[CW];
                            if (empty_tile) {
#pragma unroll
                                for (int j = 0; j < CW; ++j) own[j] = 0u;
                            } else {
                                tmem_ld_32x32b_x32(t_row + uint32_t(4 * qc), *reinterpret_cast<uint32_t(*)[32]>(own));
                                if (CW == 64)
                                    tmem_ld_32x32b_x32(t_row + uint32_t(4 * qc + 32),
                                                       *reinterpret_cast<uint32_t(*)[32]>(own + (CW == 64 ? 32 : 0)));
                                tmem_ld_wait();
                            }
                            const int col = qc * 4;
                            const bool live = ti.valid && col < cols_valid;
                            uint32_t w[32];   // the chunk's 128-byte output row
                            const uint32_t src0 = rec_u32 + uint32_t(((qc - w0) * kTileM + lrow) * 16);
                            const uint32_t sstride = uint32_t(pr) * kTileM * 16u;   // between peers' parts
#pragma unroll
                            for (int j = 0; j < C4; ++j) {
                                float4 a = make_float4(__uint_as_float(own[4 * j]), __uint_as_float(own[4 * j + 1]),
                                                       __uint_as_float(own[4 * j + 2]), __uint_as_float(own[4 * j + 3]));
                                const uint32_t sj = src0 + uint32_t(j * kTileM * 16);
                                if (csplit == 2) {
                                    // two splits: p0 + p1 == p1 + p0 (one rounding either way)
                                    const float4 b = lds_v4(sj);
                                    a.x += b.x;
                                    a.y += b.y;
                                    a.z += b.z;
                                    a.w += b.w;
                                } else {
                                    // split order s = 0, 1, ..., S - 1 with this CTA's own part at srank
                                    float4 t = srank == 0 ? a : lds_v4(sj);
#pragma unroll 1
                                    for (int sp = 1; sp < csplit; ++sp) {
                                        const float4 b =
                                            sp == srank ? a : lds_v4(sj + uint32_t(sp - (sp > srank)) * sstride);
                                        t.x += b.x;
                                        t.y += b.y;
                                        t.z += b.z;
                                        t.w += b.w;
                                    }
                                    a = t;
                                }
                                if (OUT_F32) {
                                    w[4 * j] = __float_as_uint(a.x);
                                    w[4 * j + 1] = __float_as_uint(a.y);
                                    w[4 * j + 2] = __float_as_uint(a.z);
                                    w[4 * j + 3] = __float_as_uint(a.w);
                                } else {
                                    w[2 * j] = pack_bf16x2(a.x, a.y);
                                    w[2 * j + 1] = pack_bf16x2(a.z, a.w);
                                }
                            }
                            if (!p.tma_store && live && row_ok) {
                                // no TMA stores: the row chunk's float4 columns straight to its row
#pragma unroll
                                for (int j = 0; j < C4; ++j) {
                                    if (qc + j >= w1 || col + 4 * j >= cols_valid) continue;
                                    const int64_t o = out_base + int64_t(lrow) * ld + col + 4 * j;
                                    if (OUT_F32)
                                        *reinterpret_cast<uint4 *>(static_cast<float *>(p.out) + o) =
                                            make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                                    else
                                        *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.out) + o) =
                                            make_uint2(w[2 * j], w[2 * j + 1]);
                                }
                            }
                            if (stage_out && live) {
                                // a 4 KB slab: 32 rows x 128 bytes, 128-byte swizzle (rows past the
                                // output and columns past the slice's end are clipped by the map)
                                const uint32_t slab = ostg + uint32_t((qc - w0) / C4) * 4096u;
                                const uint32_t rowp = slab + uint32_t(lane) * 128u;
#pragma unroll
                                for (int ch = 0; ch < 8; ++ch)
                                    sts_v4(rowp + uint32_t((ch ^ (lane & 7)) << 4), w[4 * ch], w[4 * ch + 1],
                                           w[4 * ch + 2], w[4 * ch + 3]);
                                fence_proxy_async_smem();
                                __syncwarp();
                                if (lane == 0) {
                                    tma_store_3d(&mapOut, slab, ti.nt * p.bn + col, ti.mt * kTileM + q * 32, ti.e);
                                    bulk_commit_group();
                                }
                                __syncwarp();
                            }
                        }
                    }
                    if (!cs_ok) break;
                    // the accumulator is read: free for the MMA warp (of the even CTA)
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        if (leader) mbar_arrive(smem_u32(&c->tempty[acc]));
                        else mbar_arrive_remote(map_to_cta(smem_u32(&c->tempty[acc]), lead));
                    }
                    // the slice is read and the slabs' stores have read them: the ring
                    // takes the next tile's copies
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
                    fence_proxy_async_smem();
                    named_bar_sync(ebar, 128);
                    if (etid == 0) mbar_arrive(smem_u32(&c->ring_free));
                    continue;
                } else {
                    if (cs_it > 0) {
                        bool okc = cluster_wait(smem_u32(&c->red_consumed), uint32_t((cs_it - 1) & 1), c, p);
                        if (!named_bar_and(ebar, 128, okc)) break;
                    }
                    // this CTA's arrival on its own red_ready, expecting the other splits' bytes
                    if (etid == 0) mbar_arrive_expect_tx(smem_u32(&c->red_ready), cs_expect);
                    cs_armed = true;
                }
                // only the float4 columns that reach the output travel
                for (int c0 = 0; c0 < 4 * nq; c0 += 32) {
                    float v[32];
                    if (empty_tile) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = 0.0f;
                    } else {
                        uint32_t r[32];
                        tmem_ld_32x32b_x32(t_row + uint32_t(c0), r);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                    }
                    // owner of the chunk's first float4 column and its place in that
                    // owner's slice: one division per 32 columns, then counting
                    int owner = (c0 >> 2) / per;
                    int rel = (c0 >> 2) - owner * per;
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const int qi = (c0 >> 2) + j4;   // float4 column of the tile
                        if (qi < nq) {
                            const uint32_t off = uint32_t(((srank * per + rel) * kTileM + lrow) * 16);
                            const float4 x = make_float4(v[4 * j4], v[4 * j4 + 1], v[4 * j4 + 2], v[4 * j4 + 3]);
                            const uint32_t dst = uint32_t(owner * PAIR + half);   // the owner's CTA of this half
                            if (owner == srank)
                                *reinterpret_cast<float4 *>(rec + off) = x;
                            else
                                st_async_v4(map_to_cta(rec_u32 + off, dst), x,
                                            map_to_cta(smem_u32(&c->red_ready), dst));
                        }
                        if (++rel == per) {
                            rel = 0;
                            ++owner;
                        }
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if (leader) mbar_arrive(smem_u32(&c->tempty[acc]));
                    else mbar_arrive_remote(map_to_cta(smem_u32(&c->tempty[acc]), lead));
                }
                named_bar_sync(ebar, 128);   // this CTA's own part of its slice is in place
                bool okr = cluster_wait(smem_u32(&c->red_ready), uint32_t(cs_it & 1), c, p);
                if (!named_bar_and(ebar, 128, okr)) break;
                cs_open = false;   // every peer's part of the slice has landed
                // my slice, summed over the splits in split order (s = 0, 1, ..., S - 1)
                constexpr bool kTr = MODE == kModeWgrad && SWAP;   // transposed output
                for (int q = q0; q < q1; ++q) {
                    const uint8_t *src = rec + (size_t(q - q0) * kTileM + lrow) * 16;
                    float4 a = *reinterpret_cast<const float4 *>(src);
#pragma unroll
                    for (int sp = 1; sp < 8; ++sp) {   // (at most 8 splits in a cluster)
                        if (sp < csplit) {
                            const float4 b = *reinterpret_cast<const float4 *>(src + size_t(sp) * per * kTileM * 16);
                            a.x += b.x;
                            a.y += b.y;
                            a.z += b.z;
                            a.w += b.w;
                        }
                    }
                    const int col = q * 4;
                    if (row_ok && ti.valid && col < cols_valid) {
                        const float vv[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const int64_t idx = kTr ? out_base + int64_t(col + q4) * ld + lrow
                                                    : out_base + int64_t(lrow) * ld + col + q4;
                            store_scalar<OUT_F32>(p.out, idx, vv[q4]);
                        }
                    }
                }
                // done with my receive buffer (a cluster's last unit needs no signal:
                // every push has landed once its owner's wait ended, and the teardown
                // cluster barrier keeps every peer alive)
                if (t + unit_step < total) {
                    named_bar_sync(ebar, 128);
                    if (etid == 0)
                        for (int j = 0; j < csplit; ++j)
                            mbar_arrive_cluster(map_to_cta(smem_u32(&c->red_consumed), j));
                }
                ++cs_it;
                continue;
            }

            // partial slots per split (deterministic mode and tail pieces), or one
            // accumulator per output tile (non-deterministic global splits)
            const bool slots = p.det || ti.tail;
            float *slot_ptr = nullptr;
            if (split) {
                slot_ptr = slots ? p.partials + ti.slot * int64_t(kTileM) * p.bn
                                 : p.partials + int64_t(ti.ticket) * kTileM * p.bn;
            }

            // full 32-row slabs of a non-split, non-transposed tile go out through
            // shared memory and TMA tensor stores (whole 128-byte lines); rows at
            // an expert's end use the masked direct stores below
            const bool tma_path = p.tma_store && ti.valid && !split && !(MODE == kModeWgrad && SWAP) &&
                                  (MODE == kModeWgrad ? q * 32 < rows_valid : q * 32 + 32 <= rows_valid);
            if (tma_path) {
                constexpr int CW = OUT_F32 ? 32 : 64;  // columns per 128-byte row
                // only chunks that exist: every staging write must be followed by its
                // committed store, or the alternating-buffer wait (all groups but the
                // newest have read their buffers) would let a write overtake a store
                for (int c0 = 0; c0 < tcw && c0 < cols_valid; c0 += CW) {
                    uint32_t w[32];
                    if (empty_tile) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) w[j] = 0u;
                    } else if (OUT_F32) {
                        tmem_ld_32x32b_x32(t_row + uint32_t(c0), w);
                        tmem_ld_wait();
                    } else {
                        uint32_t r0[32], r1[32];
                        tmem_ld_32x32b_x32(t_row + uint32_t(c0), r0);
                        tmem_ld_32x32b_x32(t_row + uint32_t(c0 + 32), r1);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            w[j] = pack_bf16x2(__uint_as_float(r0[2 * j]), __uint_as_float(r0[2 * j + 1]));
                            w[16 + j] = pack_bf16x2(__uint_as_float(r1[2 * j]), __uint_as_float(r1[2 * j + 1]));
                        }
                    }
                    const int32_t x = ti.nt * p.bn + tc0 + c0;
                    if (MODE == kModeWgrad)
                        stage_and_store<MODE>(stg_base, stg_buf, p.staging_bufs, q, lane, w, &mapOut, x,
                                              ti.mt * kTileM + q * 32, ti.e);
                    else
                        stage_and_store<MODE>(stg_base, stg_buf, p.staging_bufs, q, lane, w, &mapOut, x,
                                              ti.row0 + q * 32, 0);
                }
            }
            for (int c0 = 0; c0 < tcw && !tma_path; c0 += 32) {
                float v[32];
                if (empty_tile) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0.0f;
                } else {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(t_row + uint32_t(c0), r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                }
                if (split) {
                    // partial tile, layout [col/4][row] float4: a warp writes 512 contiguous bytes
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        float *dst = slot_ptr + (int64_t((c0 >> 2) + j4) * kTileM + lrow) * 4;
                        if (slots)
                            *reinterpret_cast<float4 *>(dst) =
                                make_float4(v[4 * j4], v[4 * j4 + 1], v[4 * j4 + 2], v[4 * j4 + 3]);
                        else
                            red_add_v4_f32(dst, v[4 * j4], v[4 * j4 + 1], v[4 * j4 + 2], v[4 * j4 + 3]);
                    }
                } else if (row_ok && c0 < cols_valid) {
                    if (MODE == kModeWgrad && SWAP) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (c0 + j < cols_valid)
                                store_scalar<OUT_F32>(p.out, out_base + int64_t(c0 + j) * ld + lrow, v[j]);
                    } else {
                        store_row32<OUT_F32>(p.out, out_base + int64_t(lrow) * ld + c0, cols_valid - c0, v);
                    }
                }
            }
            // accumulator buffer free for the MMA warp (of the even CTA of a pair)
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if (leader) mbar_arrive(smem_u32(&c->tempty[acc]));
                else mbar_arrive_remote(map_to_cta(smem_u32(&c->tempty[acc]), lead));
            }

            if (split) {
                // ticket: count this split's arrival.  Every split that then sees all
                // S partials of the tile written (the last to arrive at once, earlier
                // ones after a short bounded poll) claims 64-column slices of the tile
                // and reduces them; the last one keeps claiming until none is left, so
                // the tile is always finished and no split ever waits on work that has
                // not started.  A slice's sum is in split order, whoever computes it.
                // Claims are fetch-and-adds on the same ticket word once it holds all
                // S arrivals of this call (count - S = the slice); the next claim is
                // issued before the current slice is reduced, hiding its latency.
                __syncwarp();
                named_bar_sync(ebar, 128);
                if (etid == 0) {
                    __threadfence();
                    const uint32_t before = ticket_arrive(p.tickets + ti.ticket, c->epoch, p.status);
                    bool all_in = before == uint32_t(ti.S - 1);
                    if (!all_in && before != 0xffffffffu && p.spin_ns > 0) {
                        const uint64_t t0 = global_timer_ns();
                        while (!all_in && global_timer_ns() - t0 < p.spin_ns) {
                            const uint64_t w = ld_acquire_gpu_u64(p.tickets + ti.ticket);
                            all_in = uint32_t(w >> 32) == c->epoch && uint32_t(w & 0xffffffffu) >= uint32_t(ti.S);
                        }
                    }
                    c->last_flag = all_in;
                }
                __syncwarp();
                named_bar_sync(ebar, 128);
                const bool all_in = c->last_flag != 0;
                named_bar_sync(ebar, 128);  // everyone read last_flag before the next tile rewrites it
                if (all_in) {
                    __threadfence();
                    float *base0 = slots ? p.partials + (ti.slot - ti.s) * int64_t(kTileM) * p.bn
                                               : slot_ptr;
                    const int nsum = slots ? ti.S : 1;
                    const int64_t slot_stride = int64_t(kTileM) * p.bn;
                    const int nsl = (p.bn + 63) / 64;   // 64-column slices (16 float4 columns)
                    constexpr bool kTr = MODE == kModeWgrad && SWAP;   // transposed output
                    // (16 loads in flight; 8 in swapped kernels, which also hold
                    // the cluster reduction and otherwise pass the register limit)
                    constexpr int kCB = kTr ? 8 : 16;
                    uint64_t *tk = p.tickets + ti.ticket;
                    if (etid == 0) c->claim = int32_t(uint32_t(ticket_claim(tk)) - uint32_t(ti.S));
                    named_bar_sync(ebar, 128);
                    int sl = c->claim;
                    named_bar_sync(ebar, 128);  // everyone read the claim before it is replaced
                    while (sl >= 0 && sl < nsl) {
                        unsigned long long nxt = 0;
                        if (etid == 0) nxt = ticket_claim(tk);  // in flight while this slice is reduced
                        const int c4b = sl * 16, c4e = sl * 16 + 16 < p.bn / 4 ? sl * 16 + 16 : p.bn / 4;
                        if (nsum == 1)
                            finish_split_row<kCB, 1, OUT_F32, kTr>(base0, nsum, slot_stride, !slots, c4b, c4e, lrow,
                                                                   row_ok, cols_valid, p.out, out_base, ld);
                        else if (nsum == 2)
                            finish_split_row<kCB / 2, 2, OUT_F32, kTr>(base0, nsum, slot_stride, !slots, c4b, c4e,
                                                                       lrow, row_ok, cols_valid, p.out, out_base, ld);
                        else
                            finish_split_row<kCB / 4, 4, OUT_F32, kTr>(base0, nsum, slot_stride, !slots, c4b, c4e,
                                                                       lrow, row_ok, cols_valid, p.out, out_base, ld);
                        if (etid == 0) c->claim = int32_t(uint32_t(nxt) - uint32_t(ti.S));
                        named_bar_sync(ebar, 128);
                        sl = c->claim;
                        named_bar_sync(ebar, 128);
                    }
                }
            }
        }
        if (csplit > 0 && cs_open && etid == 0 && (PAIR == 1 || cs_armed)) {
            // left on an abort while a tile's receive phase was open: peers may
            // have pushed (or be pushing) their parts of this CTA's slice, and
            // asynchronous stores into it must land before the CTA retires.  Arm
            // the phase if this CTA had not, then wait for it with a short limit
            // (a peer that gave up before pushing never completes it; a peer
            // pushes all of its parts of a tile or none).  Pairs push only after
            // the owner armed and signalled.
            if (!cs_armed) mbar_arrive_expect_tx(smem_u32(&c->red_ready), cs_expect);
            drain_wait(smem_u32(&c->red_ready), uint32_t(cs_it & 1), 2000000ull);
        }
    } else {
        // ================== converters (router: warps 6..9) ==================
        // Thread `crow` owns A row crow of every stage -- the TMEM lane it may
        // write (warp w reaches lanes 32 (w % 4) .. + 31): its 64 FP32 values (one
        // 128-byte row in each of the two 32-column boxes, 128-byte swizzle)
        // become 32 columns of BF16 high parts and 32 of low parts in the
        // stage's A slot of tensor memory (two K elements per 32-bit column,
        // the lower index in the lower half), which the MMAs read as their A
        // operand; shared memory keeps the FP32 tile unchanged.
        const int crow = (warp & 3) * 32 + lane;
        const int sw = crow & 7;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (UnitSeq us{0, 0}; ok && warp_next_unit(us, unit0, unit_step, total, leader, lead, lane, c, p, ok);) {
            const Tile ti = decode_tile(g, us.t, t_off, t_order, t_pref, t_spref, rank);
            for (int kb = ti.kb0; kb < ti.kb1; ++kb) {
                if (!warp_wait(smem_u32(&c->full[stage]), phase, c, p)) {
                    ok = false;
                    break;
                }
                uint8_t *row_a = ring + size_t(stage) * stage_bytes + size_t(crow) * 128u;
                uint8_t *row_b = row_a + kRouterABytes / 2;
                float v[64];
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const float4 x0 = *reinterpret_cast<const float4 *>(row_a + ((ch ^ sw) << 4));
                    const float4 x1 = *reinterpret_cast<const float4 *>(row_b + ((ch ^ sw) << 4));
                    v[4 * ch] = x0.x; v[4 * ch + 1] = x0.y; v[4 * ch + 2] = x0.z; v[4 * ch + 3] = x0.w;
                    v[32 + 4 * ch] = x1.x; v[33 + 4 * ch] = x1.y; v[34 + 4 * ch] = x1.z; v[35 + 4 * ch] = x1.w;
                }
                uint32_t hi[32], lo[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    // one rounding gives both high parts; widened back exactly from their bits
                    hi[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
                    const float h0 = __uint_as_float(hi[j] << 16), h1 = __uint_as_float(hi[j] & 0xFFFF0000u);
                    lo[j] = pack_bf16x2(v[2 * j] - h0, v[2 * j + 1] - h1);      // v - hi is exact in FP32
                }
                // the stage's A slot (its last readers, the MMAs of the stage's
                // previous use, completed before the producer refilled the stage)
                const uint32_t ta = tmem_base + (uint32_t((warp & 3) * 32) << 16) + 256u + uint32_t(stage) * 64u;
                tmem_st_32x32b_x32(ta, hi);
                tmem_st_32x32b_x32(ta + 32u, lo);
                tmem_st_wait();
                // tensor-memory stores -> ordered before the MMA warp's reads
                tc_fence_before_sync();
                named_bar_sync(2, 128);
                if (warp == 6 && lane == 0) {
                    if (leader) mbar_arrive(smem_u32(&c->conv[stage]));
                    else mbar_arrive_cluster(map_to_cta(smem_u32(&c->conv[stage]), lead));
                }
                if (++stage == p.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    }

    if (warp >= 2 && (!RT || warp < 6)) {
        if (lane == 0) bulk_wait_all();  // epilogue stores complete before the CTA retires
        __syncwarp();
    }

    // ---- teardown: every role is done; release TMEM ----
    __syncwarp();
    if (cl > 1 && !early_wait) cluster_wait_acquire();  // the set-up barrier's second half
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1 && PAIR == 1) {
        tc_fence_after_sync();
        tmem_dealloc<1>(tmem_base, uint32_t(p.tmem_cols));
    }
    // no CTA leaves while a peer may still read its shared memory, write its
    // TMEM or arrive on its barriers
    if (cl > 1) cluster_sync_all();
    if (warp == 1 && PAIR == 2) {
        // both CTAs free the pair's columns together
        tc_fence_after_sync();
        tmem_dealloc<2>(tmem_base, uint32_t(p.tmem_cols));
    }
}

}  // namespace cakegg
