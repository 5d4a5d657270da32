// Paged decode attention for sm_103a (one query token per sequence).
//
// What it computes ("Q32: vLLM PagedAttention 原理" §2 and follow-up 3;
// data.6616ai.com "把虚拟内存搬进 KV Cache"): for sequence b and query head h
// (KV head g = h / G), softmax(scale * q K^T) V over the seq_lens[b] tokens
// whose K/V rows sit in the physical blocks named by block_tables[b].
//
// Work decomposition.  A "tile" is one (physical block, KV head) pair: BS
// tokens x D elements of K plus the same of V, contiguous in the pool.  The
// tiles of segment (b, g) are its n_b = ceil(len_b / BS) blocks.  All tiles of
// all segments are laid end to end (sequence-major, then KV head, then
// block) and the grid's C CTAs take contiguous ranges of that list, equal in
// a cost of tiles plus a fixed cost per segment (or, with a partition size P,
// ranges whose ends fall on multiples of P tokens).  A CTA walks its range as
// "pieces" (the part of one segment that lies in its range): a piece covering
// a whole segment is normalised and written straight to `out`; a piece of a
// segment that straddles CTAs is written as an unnormalised partial (m, l, o)
// to the workspace and counted on a per-segment counter; the CTA whose piece
// completes the count merges the segment after its own range (flash-decoding's
// reduce, with no second kernel and no CTA waiting for another):
//   M = max m_p,  out = sum e^(m_p-M) o_p / sum e^(m_p-M) l_p.
//
// CTA layout: two warps and several CTAs per SM.  The producer warp reads
// block-table entries 32 at a time (one chunk ahead) and moves each tile with
// TMA (cp.async.bulk.tensor, 128-byte swizzle, evict-first L2 hint) into an
// S-stage ring of shared-memory buffers guarded by full/empty mbarriers; the
// query rows of each piece arrive by a 1-D bulk copy.  The consumer warp
// processes the tiles in order with an online softmax (running max m, running
// sum l, fp32 accumulator o).  A piece end is a store from registers: there
// is no merge between warps and no CTA-wide barrier in the loop.
//
// Two compute paths:
//   MMA (bf16 with G >= 4, and every FP8 pool): tensor-core mma.sync m16n8k16.
//     S^T = K q^T with the 16 tokens of a half-block as M and the (padded) 8
//     query heads as N; P^T is moved into B-fragment layout with movmatrix;
//     O^T = V^T P^T with the head dimension as M.  FP8 codes are widened to f16
//     in registers (see MmaState).
//   FMA (fp32, or bf16 with G < 4): CUDA cores; lane (t, half) forms the dot
//     products of token t over half the head dimension, lanes own D/32
//     output dimensions for P V.
#pragma once

#include <cuda_fp8.h>

#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_plan.h"

namespace pa {

constexpr int kMaxGroup = 8;
constexpr int kQSlots = 2;          // query-row slots: the producer may run this many pieces ahead
constexpr int kMergeNowPieces = 3;  // an in-kernel merge of at most this many pieces may run mid-range

template <typename T>
struct ElemBytes;
template <>
struct ElemBytes<float> {
    static constexpr int value = 4;
};
template <>
struct ElemBytes<__nv_bfloat16> {
    static constexpr int value = 2;
};
template <>
struct ElemBytes<__nv_fp8_e4m3> {  // FP8 pools (OCP E4M3 codes)
    static constexpr int value = 1;
};

// Pipeline depth: about PA_STAGE_BYTES (32 KB) of tiles in flight per CTA on
// the tensor-core path and PA_STAGE_BYTES_FMA (16 KB) on the CUDA-core path,
// 2 to 16 stages.  Several CTAs share an SM: the CUDA-core path spends more
// issue slots per tile, so it keeps a shallower ring and runs twice as many
// CTAs (consumer warps) per SM for about the same bytes in flight.
#ifndef PA_STAGE_BYTES
#define PA_STAGE_BYTES 32768
#endif
#ifndef PA_STAGE_BYTES_FMA
#define PA_STAGE_BYTES_FMA 16384
#endif
#ifndef PA_STAGE_BYTES_FP8  // tensor-core path over FP8 pools, three consumer warps: 4 stages of codes
#define PA_STAGE_BYTES_FP8 32768
#endif
#ifndef PA_STAGE_BYTES_FP8_ONE  // the same with one consumer warp (8 CTAs per SM): 2 stages
#define PA_STAGE_BYTES_FP8_ONE 16384
#endif
constexpr int stages_for(int ring_bytes, int bs, int d, int e) {
    int n = ring_bytes / (2 * bs * d * e);
    return n < 2 ? 2 : (n > 16 ? 16 : n);
}

// Shared-memory layout of one CTA.  Query-row buffers are sized for the
// group size of the instantiation (GF > 0) or for the largest group.
template <typename T, int D, int BS, bool MMA, int GF, typename KV = T, int NC_ = 1>
struct Layout {
    static constexpr int E = ElemBytes<KV>::value;  // pool element bytes
    static constexpr int EQ = ElemBytes<T>::value;  // query / output element bytes
    // tiles per stage: two 16-token tiles on the tensor-core path (one handshake and one softmax
    // update per 32 tokens), one tile otherwise
    static constexpr int TPS = MMA && BS == 16 ? 2 : 1;
    static constexpr int S = stages_for(
        MMA ? (E == 1 ? (NC_ > 1 ? PA_STAGE_BYTES_FP8 : PA_STAGE_BYTES_FP8_ONE) : PA_STAGE_BYTES) : PA_STAGE_BYTES_FMA,
        BS * TPS, D, E);
    // tensor-core path over an FP8 pool: K and V codes are widened in registers
    static constexpr bool kF8 = MMA && E == 1;
    // Consumer warps (warps 0 .. NC - 1; the producer is warp NC).  Over FP8 pools the consumer,
    // which widens every code, is the bound: with NC = 3 three consumer warps take a piece's
    // stages in turn and fold their softmax states together at the piece's end.
    static constexpr int NC = NC_;
    static constexpr int kThreadsCta = 32 * (NC + 1);
    static constexpr int kProducer = NC;  // warp index
    // CTAs per SM that the register budget is planned for: that of 8 two-warp CTAs
    static constexpr int kMinCtas = kMaxCtasPerSm * 64 / kThreadsCta;
    static constexpr int GN = GF > 0 ? GF : kMaxGroup;  // query rows a q slot holds
    static constexpr int kTileBytes = BS * D * E;  // K (or V) of one tile
    static constexpr int kPanels = D * E / 128;    // 128-byte column panels per row
    static constexpr int kStageBytes = 2 * TPS * kTileBytes;  // K of its tiles, then their V
    static constexpr int kQSlotBytes = GN * D * EQ;
    static constexpr int kStagesOff = 0;
    static constexpr int kQOff = kStagesOff + S * kStageBytes;
    // CUDA-core path only: fp32 query rows (pre-scaled) and one step's weights.
    static constexpr int kQfOff = kQOff + kQSlots * kQSlotBytes;
    static constexpr int kQfBytes = MMA ? 0 : GN * D * 4;
    static constexpr int kPTileOff = kQfOff + kQfBytes;
    static constexpr int kPTileBytes = MMA ? 0 : 16 * GN * 4;
    // consumers 1 .. NC - 1 hand their softmax state to consumer 0 here at a piece's end:
    // per consumer, 4 + 4 (D / 16) floats per lane, lane-minor
    static constexpr int kCombFloats = 32 * (4 + 4 * (D / 16));
    static constexpr int kCombOff = kPTileOff + kPTileBytes;
    static constexpr int kCombBytes = (NC - 1) * kCombFloats * 4;
    static constexpr int kBarOff = kCombOff + kCombBytes;
    // Small words: [0] abort flag, [1] the consumers' stage ticket; at kPendOff the in-kernel
    // merge's two pending merges ([2][4]); at kWsumOff the lengths scan's per-warp sums (blocks,
    // then partitions: two words per warp).
    static constexpr int kMiscOff = kBarOff + (2 * S + 2 * kQSlots) * 8;
    static constexpr int kPendOff = 16;
    static constexpr int kWsumOff = kPendOff + 32;
    static constexpr int kMiscBytes = (kWsumOff + 2 * 4 * (NC + 1) + 15) / 16 * 16;
    static constexpr int kPrefixOff = kMiscOff + kMiscBytes;
    static_assert(kTileBytes % 1024 == 0, "tiles must keep 1024-byte alignment for the 128B swizzle");
    static_assert(kQSlotBytes % 16 == 0, "bulk-copy destination alignment");
    static_assert(kBarOff % 8 == 0, "mbarrier alignment");
    // dynamic shared memory for num_seqs sequences: prefix sums (two with a
    // partition size), the clamped lengths, +1 KB to align the base
    static constexpr int bytes(int num_seqs, bool fixed) {
        return kPrefixOff + (num_seqs + 1) * 4 * (fixed ? 2 : 1) + num_seqs * 4 + 1024;
    }
};

// Warp-collective wait used by both roles: every lane of the warp calls it.
// It gives up after limit_ns, or as soon as the other role has given up (the
// CTA's abort flag): the giving-up warp flags PA_DEV_WAIT_TIMEOUT and sets the
// abort flag.  After an abort the consumer releases no stage or query slot and
// the producer issues no copy, so no copy can land in a buffer that another is
// still filling; the producer then waits (full limit) for the copies it issued.
__device__ __forceinline__ bool role_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag,
                                          int32_t* status, uint64_t limit_ns = kWaitLimitNs) {
    if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
    bool ok = mbar_wait(bar, parity, limit_ns, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
        *abort_flag = 1;
        if ((threadIdx.x & 31) == 0) flag_status(status, PA_DEV_WAIT_TIMEOUT);
    }
    return ok;
}

// Several consumer warps share one stage ring; a stage's full barrier may only be waited on once
// the stage before it has been taken, so that the slot's previous fill has landed (else a
// parity wait could see the completed phase of the fill before it).  `ticket` holds the next
// stage to take.  Warp-collective, bounded like role_wait; gives up at once after an abort.
__device__ __forceinline__ bool ticket_wait(volatile int32_t* ticket, int32_t want, volatile int32_t* abort_flag,
                                            int32_t* status, uint64_t limit_ns) {
    bool ok = true;
    if (*ticket != want) {
        const uint64_t t0 = global_timer_ns();
        while (*ticket != want) {
            if (*abort_flag) {
                ok = false;
                break;
            }
            if (global_timer_ns() - t0 >= limit_ns) {
                *abort_flag = 1;
                if ((threadIdx.x & 31) == 0) flag_status(status, PA_DEV_WAIT_TIMEOUT);
                ok = false;
                break;
            }
            __nanosleep(32);
        }
    }
    return __all_sync(0xffffffffu, ok);
}


// Per-sequence blocks (and partitions) of the batch as exclusive prefix sums
// in shared memory: pref[b] (pref[B] = the total), upref likewise in
// partitions when p.partition_tiles > 0, and lens_s[b] = the clamped length.
// Run by all NT threads; wsum holds 2 * NT / 32 ints.  The caller syncs after.
template <int BS, int NT>
__device__ __forceinline__ void scan_lengths(const DecodeParams& p, bool flag_bad, int32_t* pref, int32_t* upref,
                                             int32_t* lens_s, int32_t* wsum) {
    constexpr int NW = NT / 32;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = p.num_seqs;
    const bool fixed = p.partition_tiles > 0;
    const int per = (B + NT - 1) / NT;
    const int lo = min(B, tid * per), hi = min(B, lo + per);
    int32_t nblk = 0, nprt = 0;
    for (int b = lo; b < hi; ++b) {
        const int raw_len = __ldg(p.seq_lens + b);
        if ((raw_len < 0 || raw_len > p.max_len) && flag_bad) flag_status(p.status, PA_DEV_BAD_SEQ_LEN);
        const int nb = (clamp_len(raw_len, p.max_len) + BS - 1) / BS;
        nblk += nb;
        if (fixed) nprt += (nb + p.partition_tiles - 1) / p.partition_tiles;
    }
    int32_t xb = nblk, xp = nprt;  // inclusive warp scans
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t yb = __shfl_up_sync(0xffffffffu, xb, off);
        const int32_t yp = __shfl_up_sync(0xffffffffu, xp, off);
        if (lane >= off) {
            xb += yb;
            xp += yp;
        }
    }
    if (lane == 31) {
        wsum[warp] = xb;
        wsum[NW + warp] = xp;
    }
    __syncthreads();
    int32_t ob = 0, op = 0;
    for (int w = 0; w < warp; ++w) {
        ob += wsum[w];
        op += wsum[NW + w];
    }
    int32_t rb = ob + xb - nblk, rp = op + xp - nprt;
    for (int b = lo; b < hi; ++b) {
        const int len = clamp_len(__ldg(p.seq_lens + b), p.max_len);
        const int nb = (len + BS - 1) / BS;
        lens_s[b] = len;
        pref[b] = rb;
        rb += nb;
        if (fixed) {
            upref[b] = rp;
            rp += (nb + p.partition_tiles - 1) / p.partition_tiles;
        }
    }
    if (tid == NT - 1) {
        pref[B] = ob + xb;
        if (fixed) upref[B] = op + xp;
    }
}

// A host-built plan (pa_decode_build_plan) for exactly this launch: its header must name the
// same batch, grid and split parameters, else the launch computes its own.  Every thread of
// the CTA checks the header (one cache line).
__device__ __forceinline__ bool plan_matches(const DecodeParams& p, int bs) {
    const int32_t* pl = p.plan;
    if (pl == nullptr) return false;
    return __ldg(pl + kPlanWMagic) == kPlanMagic && __ldg(pl + kPlanWNumSeqs) == p.num_seqs &&
           __ldg(pl + kPlanWGrid) == p.num_ctas && __ldg(pl + kPlanWKvHeads) == p.num_kv_heads &&
           __ldg(pl + kPlanWPartitionTiles) == p.partition_tiles && __ldg(pl + kPlanWSegUnits) == p.seg_units &&
           __ldg(pl + kPlanWBlockSize) == bs && __ldg(pl + kPlanWMaxLen) == p.max_len &&
           __ldg(pl + kPlanWMergeInKernel) == p.merge_in_kernel &&
           __ldg(pl + kPlanWMaxBlocks) == p.max_blocks_per_seq && __ldg(pl + kPlanWWaveCtas) == p.wave_ctas &&
           __ldg(pl + kPlanWWaveSkew) == p.wave_skew;
}
// The plan's prefix sums and clamped lengths go into the shared-memory arrays the scan would
// fill (pref[B + 1], then upref[B + 1] with partitions, then lens_s[B]).  Each of the NT threads
// holds kPlanPass words of a pass in registers: the first pass is loaded with the plan's record
// (plan_words_load), the later ones while the previous pass is stored.
constexpr int kPlanPass = 8;
template <int NT>
__device__ __forceinline__ void plan_words_load(const DecodeParams& p, int pass, int32_t (&v)[kPlanPass]) {
    const int n = 3 * p.num_seqs + 2;
    const int32_t* arr = p.plan + kPlanHeaderWords;
#pragma unroll
    for (int u = 0; u < kPlanPass; ++u) {
        const int w = (pass * kPlanPass + u) * NT + (int)threadIdx.x;
        v[u] = w < n ? __ldg(arr + w) : 0;
    }
}
template <int NT>
__device__ __forceinline__ void load_plan_arrays(const DecodeParams& p, int32_t (&v)[kPlanPass], int32_t* pref,
                                                 int32_t* upref, int32_t* lens_s) {
    const int B = p.num_seqs, n = 3 * B + 2;
    const bool fixed = p.partition_tiles > 0;
    for (int pass = 0; pass * kPlanPass * NT < n; ++pass) {
        int32_t nv[kPlanPass];
        plan_words_load<NT>(p, pass + 1, nv);
#pragma unroll
        for (int u = 0; u < kPlanPass; ++u) {
            const int w = (pass * kPlanPass + u) * NT + (int)threadIdx.x;
            if (w >= n) break;
            if (w <= B)
                pref[w] = v[u];
            else if (w <= 2 * B + 1) {
                if (fixed) upref[w - B - 1] = v[u];
            } else
                lens_s[w - 2 * B - 2] = v[u];
        }
#pragma unroll
        for (int u = 0; u < kPlanPass; ++u) v[u] = nv[u];
    }
}

// The plan of this launch over the scanned batch (pa_plan.h).
__device__ __forceinline__ Plan make_plan(const DecodeParams& p, const int32_t* pref, const int32_t* upref) {
    return plan_from_prefix(pref, upref, p.num_seqs, p.num_kv_heads, p.partition_tiles, p.seg_units, p.num_ctas,
                            p.wave_ctas, p.wave_skew);
}

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ float from_float<float>(float x) {
    return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Load 16 bytes of a tile row and widen to fp32 (8 bf16 or 4 fp32 values).
template <typename T>
__device__ __forceinline__ void load_chunk_f32(uint32_t addr, float* v);
template <>
__device__ __forceinline__ void load_chunk_f32<__nv_bfloat16>(uint32_t addr, float* v) {
    uint32_t r0, r1, r2, r3;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
    v[0] = bf16_lo(r0); v[1] = bf16_hi(r0); v[2] = bf16_lo(r1); v[3] = bf16_hi(r1);
    v[4] = bf16_lo(r2); v[5] = bf16_hi(r2); v[6] = bf16_lo(r3); v[7] = bf16_hi(r3);
}
template <>
__device__ __forceinline__ void load_chunk_f32<float>(uint32_t addr, float* v) {
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]) : "r"(addr));
}

// Load N consecutive elements (N * E <= 16 bytes, naturally aligned) and widen.
template <typename T, int N>
__device__ __forceinline__ void load_vec_f32(uint32_t addr, float* v) {
    if constexpr (sizeof(T) == 2) {
        if constexpr (N == 2) {
            uint32_t r;
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(addr));
            v[0] = bf16_lo(r); v[1] = bf16_hi(r);
        } else {
            static_assert(N == 4, "bf16 vector of 2 or 4");
            uint32_t r0, r1;
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
            v[0] = bf16_lo(r0); v[1] = bf16_hi(r0); v[2] = bf16_lo(r1); v[3] = bf16_hi(r1);
        }
    } else {
        if constexpr (N == 2) {
            asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v[0]), "=f"(v[1]) : "r"(addr));
        } else {
            static_assert(N == 4, "fp32 vector of 2 or 4");
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]) : "r"(addr));
        }
    }
}

// ---------------------------------------------------------------------------
// Online-softmax state of the consumer warp, per compute path
// ---------------------------------------------------------------------------

// Tensor-core path.  Thread (g = lane/4, tig = lane%4) holds the running max
// and sum of heads 2tig and 2tig+1, and O^T fragments o[mt] = rows (dims)
// 16mt+g, 16mt+g+8 x columns (heads) 2tig, 2tig+1.
// F16: operands in f16 instead of bf16 (tiles widened from an FP8 pool; the
// bf16 query rows are rounded to f16 when loaded).
// F8: K and V are E4M3 codes read straight from the stage and widened to f16 in
// registers (q is converted to f16 once per piece).  An ldmatrix over code
// pairs gives each thread four codes, and the fragments are built from them:
// - S = K q^T: a thread's four codes of a K row are four consecutive dims, so
//   a 16-dim k-step takes the dims 16 s + 4 t .. + 3 for thread quad t = lane % 4
//   instead of the usual ones (the dot product's order is free) and q's
//   fragments use the same dims.
// - O^T = V^T P^T: ldmatrix.trans gives a thread the codes of tokens 2t, 2t+1
//   at dims 16 c + 2 g and + 1; a byte permute makes the token pair of each dim
//   one f16 pair, so an m16 block's rows g and g + 8 are the dims 16 c + 2 g and
//   16 c + 2 g + 1, which the output stores undo.
template <int D, int BS, bool F8 = false>
struct MmaState {
    static constexpr bool F16 = F8;  // the MMA runs in f16 over an FP8 pool, else in bf16
    static constexpr int MT = D / 16;
    uint32_t qb[MT][2];  // B fragments of q^T per 16-dim k-step
    float m[2], l[2];
    float o[MT][4];

    __device__ static __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                    uint32_t b0, uint32_t b1) {
        if constexpr (F16)
            mma_f16_16816(d, a0, a1, a2, a3, b0, b1);
        else
            mma_bf16_16816(d, a0, a1, a2, a3, b0, b1);
    }
    __device__ static __forceinline__ uint32_t pack16(float lo, float hi) {
        if constexpr (F16)
            return pack_f16x2(lo, hi);
        else
            return pack_bf16x2(lo, hi);
    }
    __device__ static __forceinline__ float lo16(uint32_t v) { return F16 ? f16_lo(v) : bf16_lo(v); }
    __device__ static __forceinline__ float hi16(uint32_t v) { return F16 ? f16_hi(v) : bf16_hi(v); }

    __device__ __forceinline__ void reset() {
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
#pragma unroll
        for (int i = 0; i < MT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    }

    __device__ __forceinline__ void load_q(const uint8_t* qslot, int G, int lane) {
        const int g = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int s = 0; s < MT; ++s) {
            uint32_t lo = 0, hi = 0;
            if (g < G) {
                const uint32_t* row = reinterpret_cast<const uint32_t*>(qslot + (size_t)g * D * 2);
                lo = row[(F8 ? 16 * s + 4 * tig : 16 * s + 2 * tig) >> 1];
                hi = row[(F8 ? 16 * s + 4 * tig + 2 : 16 * s + 2 * tig + 8) >> 1];
                if constexpr (F16) {
                    lo = pack_f16x2(bf16_lo(lo), bf16_hi(lo));
                    hi = pack_f16x2(bf16_lo(hi), bf16_hi(hi));
                }
            }
            qb[s][0] = lo;
            qb[s][1] = hi;
        }
    }

    // S^T = K q^T for rows row0..row0+15 of a tile: acc[c] are two independent accumulation chains
    // over the k-steps, (token g, head 2tig), (g, 2tig+1), (g+8, 2tig), (g+8, 2tig+1).
    __device__ __forceinline__ void scores(uint32_t kbase, int row0, int lane, float (&acc)[2][4]) const {
#pragma unroll
        for (int c = 0; c < 2; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.f;
        const int row = row0 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int csel = lane >> 4;
        if constexpr (F8) {
            // one ldmatrix: 16 code rows x 32 dims; each thread's four codes of a
            // row are the k-slots 2t, 2t+1 (lo pair) and 2t+8, 2t+9 (hi pair)
#pragma unroll
            for (int s2 = 0; s2 < MT / 2; ++s2) {
                uint32_t r0, r1, r2, r3, a0, a1, a2, a3;
                ldmatrix_x4(kbase + tile_chunk_offset<BS>(row, 2 * s2 + csel), r0, r1, r2, r3);
                e4m3x4_to_f16x2(r0, a0, a2);
                e4m3x4_to_f16x2(r1, a1, a3);
                mma16816(acc[0], a0, a1, a2, a3, qb[2 * s2][0], qb[2 * s2][1]);
                e4m3x4_to_f16x2(r2, a0, a2);
                e4m3x4_to_f16x2(r3, a1, a3);
                mma16816(acc[1], a0, a1, a2, a3, qb[2 * s2 + 1][0], qb[2 * s2 + 1][1]);
            }
        } else {
#pragma unroll
            for (int s = 0; s < MT; ++s) {
                uint32_t a0, a1, a2, a3;
                ldmatrix_x4(kbase + tile_chunk_offset<BS>(row, 2 * s + csel), a0, a1, a2, a3);
                mma16816(acc[s & 1], a0, a1, a2, a3, qb[s][0], qb[s][1]);
            }
        }
    }

    // O^T += V^T P^T for rows row0..row0+15 of a tile; b0, b1: P^T as B fragments.  MASK: some
    // of the 16 rows lie past the sequence end (a tile that is not full); only then are the V
    // operands masked, which on the FP8 path saves a quarter of the ALU work per 16 tokens.
    template <bool MASK>
    __device__ __forceinline__ void accumulate_pv_m(uint32_t vbase, int row0, int valid, uint32_t b0, uint32_t b1,
                                                    int lane) {
        const int tig = lane & 3;
        uint32_t m01 = 0xffffffffu, m89 = 0xffffffffu;
        if (MASK) {  // zero V rows past the sequence end (their slots may hold anything)
            m01 = (2 * tig < valid ? 0x0000ffffu : 0u) | (2 * tig + 1 < valid ? 0xffff0000u : 0u);
            m89 = (2 * tig + 8 < valid ? 0x0000ffffu : 0u) | (2 * tig + 9 < valid ? 0xffff0000u : 0u);
        }
        if constexpr (F8) {
            // one ldmatrix.trans: registers (tokens 0-7, chunk c), (8-15, c), (0-7, c+1), (8-15, c+1)
            const int row = row0 + (lane & 7) + (((lane >> 3) & 1) << 3);
            const int csel = lane >> 4;
#pragma unroll
            for (int i2 = 0; i2 < MT / 2; ++i2) {
                uint32_t r0, r1, r2, r3, a0, a1, a2, a3;
                ldmatrix_x4_trans(vbase + tile_chunk_offset<BS>(row, 2 * i2 + csel), r0, r1, r2, r3);
                e4m3x4_to_f16x2(__byte_perm(r0, 0, 0x3120), a0, a1);  // even dim, odd dim; tokens 2t, 2t+1
                e4m3x4_to_f16x2(__byte_perm(r1, 0, 0x3120), a2, a3);  // same dims, tokens 2t+8, 2t+9
                mma16816(o[2 * i2], a0 & m01, a1 & m01, a2 & m89, a3 & m89, b0, b1);
                e4m3x4_to_f16x2(__byte_perm(r2, 0, 0x3120), a0, a1);
                e4m3x4_to_f16x2(__byte_perm(r3, 0, 0x3120), a2, a3);
                mma16816(o[2 * i2 + 1], a0 & m01, a1 & m01, a2 & m89, a3 & m89, b0, b1);
            }
        } else {
            const int row = row0 + (lane & 7) + ((lane >> 4) << 3);
            const int csel = (lane >> 3) & 1;
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                uint32_t a0, a1, a2, a3;
                ldmatrix_x4_trans(vbase + tile_chunk_offset<BS>(row, 2 * i + csel), a0, a1, a2, a3);
                mma16816(o[i], a0 & m01, a1 & m01, a2 & m89, a3 & m89, b0, b1);
            }
        }
    }

    __device__ __forceinline__ void accumulate_pv(uint32_t vbase, int row0, int valid, uint32_t b0, uint32_t b1,
                                                  int lane) {
        if (valid < 16)
            accumulate_pv_m<true>(vbase, row0, valid, b0, b1, lane);
        else
            accumulate_pv_m<false>(vbase, row0, valid, b0, b1, lane);
    }

    // Base-2 scores of one 16-token step: (token g, head 2tig), (g, 2tig+1), (g+8, 2tig), (g+8, 2tig+1),
    // -inf past `valid`.
    __device__ static __forceinline__ void base2(const float (&acc)[2][4], int valid, float scale_log2, int lane,
                                                 float (&x)[4]) {
        const int g = lane >> 2;
        const bool v0 = g < valid, v1 = g + 8 < valid;
        x[0] = v0 ? (acc[0][0] + acc[1][0]) * scale_log2 : -INFINITY;
        x[1] = v0 ? (acc[0][1] + acc[1][1]) * scale_log2 : -INFINITY;
        x[2] = v1 ? (acc[0][2] + acc[1][2]) * scale_log2 : -INFINITY;
        x[3] = v1 ? (acc[0][3] + acc[1][3]) * scale_log2 : -INFINITY;
    }

    // Online-softmax update over the scores of n steps (n = 1 or 2); P[s][0..1] receive step s's
    // weights, packed as the MMA's A operand rows (token g, token g+8).
    template <int N>
    __device__ __forceinline__ void softmax(const float (&x)[N][4], uint32_t (&P)[N][2]) {
        float mx0 = fmaxf(x[0][0], x[0][2]), mx1 = fmaxf(x[0][1], x[0][3]);
#pragma unroll
        for (int s = 1; s < N; ++s) {
            mx0 = fmaxf(mx0, fmaxf(x[s][0], x[s][2]));
            mx1 = fmaxf(mx1, fmaxf(x[s][1], x[s][3]));
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
        const float al0 = exp2f(m[0] - mn0), al1 = exp2f(m[1] - mn1);
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int s = 0; s < N; ++s) {
            P[s][0] = pack16(exp2f(x[s][0] - mn0), exp2f(x[s][1] - mn1));
            P[s][1] = pack16(exp2f(x[s][2] - mn0), exp2f(x[s][3] - mn1));
            // the sum uses the rounded weights that P V uses
            s0 += lo16(P[s][0]) + lo16(P[s][1]);
            s1 += hi16(P[s][0]) + hi16(P[s][1]);
        }
        l[0] = l[0] * al0 + s0;
        l[1] = l[1] * al1 + s1;
        m[0] = mn0;
        m[1] = mn1;
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            o[i][0] *= al0;
            o[i][1] *= al1;
            o[i][2] *= al0;
            o[i][3] *= al1;
        }
    }

    // One 16-token step: rows row0..row0+15 of the tile, `valid` of them real.
    __device__ __forceinline__ void step(uint32_t kbase, uint32_t vbase, int row0, int valid, float scale_log2,
                                         int lane) {
        float acc[2][4], x[1][4];
        uint32_t P[1][2];
        scores(kbase, row0, lane, acc);
        base2(acc, valid, scale_log2, lane, x[0]);
        softmax<1>(x, P);
        accumulate_pv(vbase, row0, valid, movmatrix_trans(P[0][0]), movmatrix_trans(P[0][1]), lane);
    }

    // Two 16-token steps with one softmax update: their score chains are independent, and the
    // running max, sum and the rescale of O are done once for 32 tokens.
    __device__ __forceinline__ void step2(uint32_t kbase_a, uint32_t vbase_a, int row0_a, int valid_a,
                                          uint32_t kbase_b, uint32_t vbase_b, int row0_b, int valid_b,
                                          float scale_log2, int lane) {
        float acc_a[2][4], acc_b[2][4], x[2][4];
        uint32_t P[2][2];
        scores(kbase_a, row0_a, lane, acc_a);
        scores(kbase_b, row0_b, lane, acc_b);
        base2(acc_a, valid_a, scale_log2, lane, x[0]);
        base2(acc_b, valid_b, scale_log2, lane, x[1]);
        softmax<2>(x, P);
        accumulate_pv(vbase_a, row0_a, valid_a, movmatrix_trans(P[0][0]), movmatrix_trans(P[0][1]), lane);
        accumulate_pv(vbase_b, row0_b, valid_b, movmatrix_trans(P[1][0]), movmatrix_trans(P[1][1]), lane);
    }

    // Head dims of accumulator rows g and g + 8 of m16 block i.
    __device__ static __forceinline__ int dim_lo(int i, int g) { return F8 ? 16 * i + 2 * g : 16 * i + g; }
    __device__ static __forceinline__ int dim_hi(int i, int g) { return F8 ? 16 * i + 2 * g + 1 : 16 * i + g + 8; }

    // This lane's state as 4 + 4 MT floats at scr[f * 32 + lane] (another consumer warp of the
    // CTA folds it in with combine(); both warps hold the same fragments in the same lanes).
    __device__ __forceinline__ void save(float* scr, int lane) const {
        scr[lane] = m[0];
        scr[32 + lane] = m[1];
        scr[64 + lane] = l[0];
        scr[96 + lane] = l[1];
#pragma unroll
        for (int i = 0; i < MT; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) scr[(4 + 4 * i + j) * 32 + lane] = o[i][j];
    }
    // Fold a saved state (same tokens' heads, other tokens) into this one: the online-softmax
    // merge of two partial states.  A side that saw no token has m = -inf and weighs 0.
    __device__ __forceinline__ void combine(const float* scr, int lane) {
        const float om0 = scr[lane], om1 = scr[32 + lane];
        const float n0 = fmaxf(m[0], om0), n1 = fmaxf(m[1], om1);
        const float a0 = n0 == -INFINITY ? 0.f : exp2f(m[0] - n0), b0 = n0 == -INFINITY ? 0.f : exp2f(om0 - n0);
        const float a1 = n1 == -INFINITY ? 0.f : exp2f(m[1] - n1), b1 = n1 == -INFINITY ? 0.f : exp2f(om1 - n1);
        l[0] = l[0] * a0 + scr[64 + lane] * b0;
        l[1] = l[1] * a1 + scr[96 + lane] * b1;
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            o[i][0] = o[i][0] * a0 + scr[(4 + 4 * i) * 32 + lane] * b0;
            o[i][1] = o[i][1] * a1 + scr[(5 + 4 * i) * 32 + lane] * b1;
            o[i][2] = o[i][2] * a0 + scr[(6 + 4 * i) * 32 + lane] * b0;
            o[i][3] = o[i][3] * a1 + scr[(7 + 4 * i) * 32 + lane] * b1;
        }
        m[0] = n0;
        m[1] = n1;
    }

    // Sum the running sums over the 8 token rows (lanes with the same tig).
    __device__ __forceinline__ void finish() {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
            l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
        }
    }

    // Normalised output rows; `o_rows` points at out[b][h*G][0].
    // oscale multiplies the output (the V scale of an FP8 pool, else 1).
    template <typename T>
    __device__ __forceinline__ void store_out(T* o_rows, int G, int lane, float oscale) const {
        const int g = lane >> 2, h0 = 2 * (lane & 3), h1 = h0 + 1;
        const float r0 = oscale / l[0], r1 = oscale / l[1];
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            const int dl = dim_lo(i, g), dh = dim_hi(i, g);
            if (h0 < G) {
                o_rows[h0 * D + dl] = from_float<T>(o[i][0] * r0);
                o_rows[h0 * D + dh] = from_float<T>(o[i][2] * r0);
            }
            if (h1 < G) {
                o_rows[h1 * D + dl] = from_float<T>(o[i][1] * r1);
                o_rows[h1 * D + dh] = from_float<T>(o[i][3] * r1);
            }
        }
    }

    // Unnormalised partial: slot = [G][D] o, then [G] (m, l).
    __device__ __forceinline__ void store_partial(float* slot, int G, int lane) const {
        const int g = lane >> 2, h0 = 2 * (lane & 3), h1 = h0 + 1;
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            const int dl = dim_lo(i, g), dh = dim_hi(i, g);
            if (h0 < G) {
                slot[h0 * D + dl] = o[i][0];
                slot[h0 * D + dh] = o[i][2];
            }
            if (h1 < G) {
                slot[h1 * D + dl] = o[i][1];
                slot[h1 * D + dh] = o[i][3];
            }
        }
        if (g == 0) {
            if (h0 < G) { slot[G * D + 2 * h0] = m[0]; slot[G * D + 2 * h0 + 1] = l[0]; }
            if (h1 < G) { slot[G * D + 2 * h1] = m[1]; slot[G * D + 2 * h1 + 1] = l[1]; }
        }
    }
};

// CUDA-core path.  Lane = (token t = lane & 15, half = lane >> 4) for the dot
// products; lane owns output dims [lane * VEC, lane * VEC + VEC) for P V.
// GF > 0 fixes the query heads per KV head at compile time (no per-head
// predication); GF == 0 handles any G <= 8 at run time.
template <typename T, int D, int BS, int GF>
struct FmaState {
    static constexpr int E = ElemBytes<T>::value;
    static constexpr int VEC = D / 32;
    static constexpr int EPC = 16 / E;              // elements per 16-byte chunk
    static constexpr int HALF_CHUNKS = D * E / 32;  // chunks per half row
    static constexpr int GN = GF > 0 ? GF : kMaxGroup;
    float m[GN], l[GN];
    float o[GN][VEC];

    __device__ __forceinline__ static bool active(int g, int G) { return GF > 0 || g < G; }

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int g = 0; g < GN; ++g) {
            m[g] = -INFINITY;
            l[g] = 0.f;
#pragma unroll
            for (int v = 0; v < VEC; ++v) o[g][v] = 0.f;
        }
    }

    __device__ __forceinline__ void pv_token(uint32_t vbase, int row, int byte0, const float* ptile_row, int G) {
        float vv[VEC];
        load_vec_f32<T, VEC>(vbase + tile_chunk_offset<BS>(row, byte0 >> 4) + (byte0 & 15), vv);
#pragma unroll
        for (int g = 0; g < GN; ++g) {
            if (active(g, G)) {
                const float pw = ptile_row[g];
#pragma unroll
                for (int v = 0; v < VEC; ++v) o[g][v] = fmaf(pw, vv[v], o[g][v]);
            }
        }
    }

    // qf: [G][D] fp32 query rows pre-multiplied by scale*log2(e); ptile: [16][GN] weights of one step.
    __device__ __forceinline__ void step(uint32_t kbase, uint32_t vbase, int row0, int valid, int G,
                                         const float* qf, float* ptile, int lane) {
        const int t = lane & 15, half = lane >> 4;
        float acc[GN][2];  // two chains per head (even / odd chunks)
#pragma unroll
        for (int g = 0; g < GN; ++g) acc[g][0] = acc[g][1] = 0.f;
        const int row = row0 + t;
#pragma unroll
        for (int cc = 0; cc < HALF_CHUNKS; ++cc) {
            const int chunk = half * HALF_CHUNKS + cc;
            float kv[EPC];
            load_chunk_f32<T>(kbase + tile_chunk_offset<BS>(row, chunk), kv);
#pragma unroll
            for (int g = 0; g < GN; ++g) {
                if (active(g, G)) {
                    const float4* qp = reinterpret_cast<const float4*>(qf + g * D + chunk * EPC);
#pragma unroll
                    for (int e4 = 0; e4 < EPC / 4; ++e4) {
                        const float4 qv = qp[e4];
                        float& a = acc[g][cc & 1];
                        a = fmaf(qv.x, kv[4 * e4 + 0], a);
                        a = fmaf(qv.y, kv[4 * e4 + 1], a);
                        a = fmaf(qv.z, kv[4 * e4 + 2], a);
                        a = fmaf(qv.w, kv[4 * e4 + 3], a);
                    }
                }
            }
        }
        float alpha[GN];
#pragma unroll
        for (int g = 0; g < GN; ++g) {
            alpha[g] = 1.f;
            if (active(g, G)) {
                float x = acc[g][0] + acc[g][1];
                x += __shfl_xor_sync(0xffffffffu, x, 16);
                x = t < valid ? x : -INFINITY;
                float mx = x;
#pragma unroll
                for (int off = 1; off < 16; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                const float mn = fmaxf(m[g], mx);
                alpha[g] = exp2f(m[g] - mn);
                const float pw = exp2f(x - mn);
                float sum = pw;
#pragma unroll
                for (int off = 1; off < 16; off <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
                l[g] = l[g] * alpha[g] + sum;
                m[g] = mn;
                if (half == 0) ptile[t * GN + g] = pw;
            }
        }
        __syncwarp();
#pragma unroll
        for (int g = 0; g < GN; ++g)
#pragma unroll
            for (int v = 0; v < VEC; ++v) o[g][v] *= alpha[g];
        const int byte0 = lane * VEC * E;
        if (valid == 16) {
#pragma unroll
            for (int tt = 0; tt < 16; ++tt) pv_token(vbase, row0 + tt, byte0, ptile + tt * GN, G);
        } else {
            for (int tt = 0; tt < valid; ++tt) pv_token(vbase, row0 + tt, byte0, ptile + tt * GN, G);
        }
        __syncwarp();
    }

    // Normalised output rows; `o_rows` points at out[b][h*G][0].  m and l are
    // the same in every lane (reduced by shuffles in step()).
    template <typename TO>
    __device__ __forceinline__ void store_out(TO* o_rows, int G, int lane, float oscale) const {
#pragma unroll
        for (int g = 0; g < GN; ++g) {
            if (active(g, G)) {
                const float r = oscale / l[g];
#pragma unroll
                for (int v = 0; v < VEC; ++v) o_rows[g * D + lane * VEC + v] = from_float<TO>(o[g][v] * r);
            }
        }
    }

    // Unnormalised partial: slot = [G][D] o, then [G] (m, l).
    __device__ __forceinline__ void store_partial(float* slot, int G, int lane) const {
#pragma unroll
        for (int g = 0; g < GN; ++g) {
            if (active(g, G)) {
#pragma unroll
                for (int v = 0; v < VEC; ++v) slot[g * D + lane * VEC + v] = o[g][v];
                if (lane == 0) {
                    slot[G * D + 2 * g] = m[g];
                    slot[G * D + 2 * g + 1] = l[g];
                }
            }
        }
    }
};

// Partial slot of piece cc of a split segment whose first piece is in CTA ca.
// A split segment's first piece is the last piece of its CTA's range (slot 1);
// every later piece starts its CTA's range (slot 0).  A CTA's two slots are
// never both needed by one piece.
__device__ __forceinline__ const float* piece_slot(const float* partials, size_t slot_floats, int cc, int ca) {
    return partials + (size_t)(2 * cc + (cc == ca ? 1 : 0)) * slot_floats;
}

// 16 output elements (fp32 sums times sc) to 16-byte-aligned global memory.
template <typename T>
__device__ __forceinline__ void store16(T* dst, const float (&a)[16], float sc) {
    if constexpr (std::is_same<T, float>::value) {
        float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
        for (int v = 0; v < 4; ++v) d[v] = make_float4(a[4 * v] * sc, a[4 * v + 1] * sc, a[4 * v + 2] * sc, a[4 * v + 3] * sc);
    } else {
        uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int v = 0; v < 2; ++v)
            d[v] = make_uint4(pack_bf16x2(a[8 * v] * sc, a[8 * v + 1] * sc), pack_bf16x2(a[8 * v + 2] * sc, a[8 * v + 3] * sc),
                              pack_bf16x2(a[8 * v + 4] * sc, a[8 * v + 5] * sc), pack_bf16x2(a[8 * v + 6] * sc, a[8 * v + 7] * sc));
    }
}

// Merge of one split segment by a group of lps lanes (sl = this lane's index
// in the group), from the pieces' partial slots in global memory (read from
// L2, once every piece is visible: its CTA released its stores before counting
// the piece in, or the decode grid that wrote them has finished):
//   M = max_p m_p,   out = sum_p e^(m_p-M) o_p / sum_p e^(m_p-M) l_p.
// Each lane owns 16 consecutive output elements of one head per pass of
// 16 * lps elements and folds that head's max and sum itself, pieces in order,
// four at a time: their (m, l) loads in flight together, then XB pieces' o
// loads at a time (XB = 4 or 1: fewer registers).  The arithmetic does not
// depend on XB, so every merge of a segment gives the same bits.
template <typename T, int D, int XB, bool STORE = true>
__device__ __forceinline__ void merge_pieces(const float* partials, size_t slot_floats, T* orow, int ca, int np, int G,
                                             int sl, int lps, float oscale) {
    static_assert(XB == 1 || XB == 4, "o loads in flight: 1 or 4 pieces");
    const int nel = G * D;
    for (int e0 = sl * 16; e0 < nel; e0 += 16 * lps) {
        const int ml = nel + 2 * (e0 / D);  // (m, l) of this lane's head within a slot
        float mrun = -INFINITY, lrun = 0.f, a[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) a[k] = 0.f;
        for (int i0 = 0; i0 < np; i0 += 4) {
            float2 m_l[4];
            float4 x[XB][4];
            auto load_o = [&](int i) {  // o of pieces i .. i + XB - 1 of this group
#pragma unroll
                for (int j = 0; j < XB; ++j)
                    if (i0 + i + j < np) {
                        const float* sp = piece_slot(partials, slot_floats, ca + i0 + i + j, ca);
#pragma unroll
                        for (int v = 0; v < 4; ++v) x[j][v] = __ldcg(reinterpret_cast<const float4*>(sp + e0) + v);
                    }
            };
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (i0 + i < np)
                    m_l[i] = __ldcg(reinterpret_cast<const float2*>(piece_slot(partials, slot_floats, ca + i0 + i, ca) + ml));
            load_o(0);
            float mc = mrun;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (i0 + i < np) mc = fmaxf(mc, m_l[i].x);
            const float resc = exp2f(mrun - mc);  // 0 for the first four pieces
            lrun *= resc;
#pragma unroll
            for (int k = 0; k < 16; ++k) a[k] *= resc;
#pragma unroll
            for (int i = 0; i < 4; i += XB) {
                if (i > 0) load_o(i);
#pragma unroll
                for (int j = 0; j < XB; ++j) {
                    if (i0 + i + j < np) {
                        const float w = exp2f(m_l[i + j].x - mc);
                        lrun = fmaf(w, m_l[i + j].y, lrun);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            a[4 * v] = fmaf(w, x[j][v].x, a[4 * v]), a[4 * v + 1] = fmaf(w, x[j][v].y, a[4 * v + 1]);
                            a[4 * v + 2] = fmaf(w, x[j][v].z, a[4 * v + 2]), a[4 * v + 3] = fmaf(w, x[j][v].w, a[4 * v + 3]);
                        }
                    }
                }
            }
            mrun = mc;
        }
        if constexpr (STORE) store16(orow + e0, a, __fdividef(oscale, lrun));  // lrun >= 1: the largest piece max weighs 1
        else asm volatile("" ::"f"(a[0]), "f"(a[15]), "f"(lrun));  // keep the dry run's arithmetic
    }
}

// GPU-scope acquire-release fence: a release before a relaxed atomic publishes this thread's
// earlier writes (and those a barrier ordered before it); an acquire after a relaxed atomic makes
// the writes its value was published with visible to this thread's later reads.
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
// IKM: the in-kernel merge is compiled in (it runs when p.merge_in_kernel is set).
template <typename T, int D, int BS, bool MMA, int GF, typename KV, bool IKM, int NC>
__device__ __forceinline__ void decode_body(const DecodeParams& p, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v) {
    using L = Layout<T, D, BS, MMA, GF, KV, NC>;
    constexpr int S = L::S;
    constexpr int E = L::E;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_s - raw_s);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = p.num_seqs, Hkv = p.num_kv_heads, C = p.num_ctas, c = blockIdx.x;
    const int G = GF > 0 ? GF : p.group;  // query heads per KV head
    const bool fixed = p.partition_tiles > 0;
    int32_t* pref = reinterpret_cast<int32_t*>(base + L::kPrefixOff);
    int32_t* upref = pref + (B + 1);
    int32_t* lens_s = upref + (fixed ? B + 1 : 0);  // clamped seq_lens
    volatile int32_t* misc = reinterpret_cast<volatile int32_t*>(base + L::kMiscOff);
    int32_t* wsum = reinterpret_cast<int32_t*>(base + L::kMiscOff + L::kWsumOff);  // per warp: blocks, then partitions
    const uint32_t bar0 = base_s + L::kBarOff;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto qfull_bar = [&](int i) { return bar0 + 8u * (2 * S + i); };
    auto qempty_bar = [&](int i) { return bar0 + 8u * (2 * S + kQSlots + i); };

    // the producer's tensor maps and cache policy, requested before the plan is known
    uint64_t policy = 0;
    if (warp == L::kProducer) {
        if (lane == 0) {
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
        }
        policy = policy_evict_first();
    }
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int i = 0; i < kQSlots; ++i) {
            mbar_init(qfull_bar(i), 1);
            mbar_init(qempty_bar(i), L::NC);  // every consumer warp has read the rows
        }
        fence_barrier_init();
        misc[0] = 0;  // abort flag
        misc[1] = 0;  // the next ring stage a consumer warp may take (several consumer warps)
    }

    // With a host-built plan the lengths scan, the range searches and the first table chunk's
    // fetch are replaced by loads from the plan.  The host checked that the plan holds this
    // launch's words, so the header, this CTA's record and the arrays' first pass are loaded in
    // one round trip, before the header is compared; a plan for another launch is then unused.
    bool planned = false;
    int32_t rec = 0, first_chunk = 0;  // lane < 8: the CTA's record word `lane`; all: its first chunk
    int32_t pw[kPlanPass];
    if (p.plan != nullptr) {
        const int32_t* r = p.plan + plan_rec_off(B, c);
        if (lane < kRecFirst) rec = __ldg(r + lane);
        first_chunk = __ldg(r + kRecFirst + lane);
        plan_words_load<L::kThreadsCta>(p, 0, pw);
        planned = plan_matches(p, BS);
    }
    if (planned)
        load_plan_arrays<L::kThreadsCta>(p, pw, pref, upref, lens_s);
    else
        scan_lengths<BS, L::kThreadsCta>(p, c == 0, pref, upref, lens_s, wsum);
    __syncthreads();

    const Plan P = make_plan(p, pref, upref);
    // a programmatic dependent that follows on the stream may start its prologue now; it waits
    // for this grid to finish before it reads what the grid writes
    if (tid == 0) pdl_launch_dependents();
    const bool works = P.T > 0 && c < P.C;
    // the two ends of the range are two independent searches: lanes 0 and 1 of
    // each warp run one each; lane 1's also gives the start of the segment the
    // range ends inside (the walk's rotation point)
    int64_t tb = 0, split = -1;
    int seqh = 0;
    if (!planned && works && lane < 2) tb = P.cta_start(c + lane, &split, &seqh);
    const bool merge_here = IKM && p.merge_in_kernel;
    const int64_t t0 = planned ? __shfl_sync(0xffffffffu, rec, kRecT0) : __shfl_sync(0xffffffffu, tb, 0);
    const int64_t t1 = planned ? __shfl_sync(0xffffffffu, rec, kRecT1) : __shfl_sync(0xffffffffu, tb, 1);
    const int seq0 = planned ? __shfl_sync(0xffffffffu, rec, kRecSeq0) : __shfl_sync(0xffffffffu, seqh, 0);
    const int seq1 = planned ? __shfl_sync(0xffffffffu, rec, kRecSeq1) : __shfl_sync(0xffffffffu, seqh, 1);
    const int64_t ta = planned ? __shfl_sync(0xffffffffu, rec, kRecTa)
                               : __shfl_sync(0xffffffffu, merge_here ? split : -1, 1);
    const int Hq = p.num_q_heads;
    // one partial slot: [G][D] unnormalised o, then [G] (m, l)
    const size_t slot_floats = partial_slot_floats(G, D);

    if (warp == L::kProducer) {
        // =========================== producer ===========================
        // (the tensor maps were prefetched at the kernel's start)
        const uint32_t q_bytes = (uint32_t)(G * D * L::EQ);
        uint32_t k = 0, pi = 0, k_issued = 0, pi_issued = 0;
        // Walk the range in chunks of up to 32 tiles of one piece.  The block-table
        // entries of the next chunk (of this piece or of the next one) are loaded
        // before this chunk's tiles are issued, so their latency overlaps the issue.
        PieceIter<IKM> it;
        it.init(P, t0, t1, ta, seq0, seq1);
        int b = 0, h = 0, j0 = 0, j1 = 0, nb_ = 0, nh = 0, nj0 = 0, nj1 = 0;
        bool have = it.next(P, b, h, j0, j1);
        bool have_next = have && it.next(P, nb_, nh, nj0, nj1);
        auto table_chunk = [&](int bb, int jfrom, int jend) -> int32_t {
            return lane < jend - jfrom && lane < 32 ? __ldg(p.block_tables + (size_t)bb * p.max_blocks_per_seq + jfrom + lane)
                                                    : 0;
        };
        int32_t blk_cur = have ? (planned ? first_chunk : table_chunk(b, j0, j1)) : 0;
        // Everything above reads only seq_lens and block_tables, which the append and
        // copy kernels of this library never write; pool and query reads wait for the
        // preceding kernel (launched as a programmatic dependent, see pa_api.cu).
        pdl_wait_prerequisites();
        int jb = j0;
        while (have) {
            if (jb == j0) {  // first chunk of a piece: its query rows
                const int qs = pi % kQSlots;
                if (role_wait(qempty_bar(qs), ((pi / kQSlots) & 1) ^ 1, misc, p.status)) {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(qfull_bar(qs), q_bytes);
                        const uint8_t* src = static_cast<const uint8_t*>(p.q) + ((size_t)b * Hq + (size_t)h * G) * D * L::EQ;
                        bulk_load(base_s + L::kQOff + qs * L::kQSlotBytes, src, q_bytes, qfull_bar(qs));
                    }
                    pi_issued = pi + 1;
                }
            }
            const int n = min(32, j1 - jb);
            const bool more_here = jb + 32 < j1;
            int32_t blk_nxt = 0;
            if (more_here)
                blk_nxt = table_chunk(b, jb + 32, j1);
            else if (have_next)
                blk_nxt = table_chunk(nb_, nj0, nj1);
            // stages of TPS consecutive tiles of the piece (a chunk holds an even number of them
            // except at the piece's end, so the pairs are tiles 2m, 2m + 1 from the piece start)
            for (int i = 0; i < n; i += L::TPS) {
                const int nt = min(L::TPS, n - i);
                int32_t bids[L::TPS];
#pragma unroll
                for (int t = 0; t < L::TPS; ++t) {
                    int32_t bid = __shfl_sync(0xffffffffu, blk_cur, (i + t) & 31);
                    if (t < nt && (bid < 0 || bid >= p.num_blocks)) {  // warp-uniform
                        if (lane == 0) flag_status(p.status, PA_DEV_BAD_BLOCK_ID);
                        bid = 0;
                    }
                    bids[t] = bid;
                }
                const int st = k % S;
                if (role_wait(empty_bar(st), ((k / S) & 1) ^ 1, misc, p.status)) {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(full_bar(st), (uint32_t)(nt * 2 * L::kTileBytes));
                        const uint32_t ks = base_s + L::kStagesOff + st * L::kStageBytes;
#pragma unroll
                        for (int t = 0; t < L::TPS; ++t) {
                            if (t < nt) {
                                const int32_t y = (bids[t] * Hkv + h) * BS;
#pragma unroll
                                for (int pn = 0; pn < L::kPanels; ++pn) {
                                    tma_load_2d(ks + t * L::kTileBytes + pn * BS * 128, &tmap_k, pn * (128 / E), y,
                                                full_bar(st), policy);
                                    tma_load_2d(ks + (L::TPS + t) * L::kTileBytes + pn * BS * 128, &tmap_v,
                                                pn * (128 / E), y, full_bar(st), policy);
                                }
                            }
                        }
                    }
                    k_issued = k + 1;
                }
                ++k;
            }
            if (more_here) {
                jb += 32;
            } else {
                ++pi;
                b = nb_, h = nh, j0 = nj0, j1 = nj1;
                jb = j0;
                have = have_next;
                have_next = have && it.next(P, nb_, nh, nj0, nj1);
            }
            blk_cur = blk_nxt;
        }
        // never leave the CTA with copies still landing in its shared memory
        for (uint32_t kk = k_issued > (uint32_t)S ? k_issued - S : 0; kk < k_issued; ++kk)
            mbar_wait(full_bar(kk % S), (kk / S) & 1);
        for (uint32_t qq = pi_issued > (uint32_t)kQSlots ? pi_issued - kQSlots : 0; qq < pi_issued; ++qq)
            mbar_wait(qfull_bar(qq % kQSlots), (qq / kQSlots) & 1);
    } else if (warp < L::NC) {
        // =========================== consumers ===========================
        // Consumer warp cw takes the stages kk with kk % NC == cw; at a piece's end the others
        // hand their softmax state to consumer 0, which finishes the piece.
        const int cw = warp;
        // `out` may be read or written by the preceding kernel on the stream: wait
        // for it before the first store (the consumer's first query wait comes
        // after the producer's own, so this costs nothing), then zero the outputs
        // of empty sequences
        pdl_wait_prerequisites();
        for (int bb = c; cw == 0 && bb < B; bb += C) {
            if (pref[bb + 1] == pref[bb]) {
                T* o = static_cast<T*>(p.out) + (size_t)bb * Hq * D;
                for (int e = lane; e < Hq * D; e += 32) o[e] = from_float<T>(0.f);
            }
        }
        float* qf = reinterpret_cast<float*>(base + L::kQfOff);
        float* ptile = reinterpret_cast<float*>(base + L::kPTileOff);
        typename std::conditional<MMA, MmaState<D, BS, L::kF8>, FmaState<KV, D, BS, GF>>::type st;
        uint32_t k = 0, pi = 0;
        // In-kernel merges this CTA completes wait for the end of its range when they would
        // otherwise come last (its last piece) or take many round trips (more than
        // kMergeNowPieces pieces): lane 0 notes (b, h, ca, np) of at most two (slot 0 and
        // slot 1) in shared memory, np = 0 for none.
        int32_t* pend = reinterpret_cast<int32_t*>(base + L::kMiscOff + L::kPendOff);  // [2][4]
        if (IKM && cw == 0 && lane == 0) pend[3] = pend[7] = 0;
        float* comb = reinterpret_cast<float*>(base + L::kCombOff);
        PieceIter<IKM> it;
        it.init(P, t0, t1, ta, seq0, seq1);
        int b, h, j0, j1;
        while (it.next(P, b, h, j0, j1)) {
            const int qs = pi % kQSlots;
            const uint8_t* qslot = base + L::kQOff + qs * L::kQSlotBytes;
            const bool qok = role_wait(qfull_bar(qs), (pi / kQSlots) & 1, misc, p.status, p.wait_limit_ns);
            if constexpr (MMA) {
                if (qok) st.load_q(qslot, G, lane);
            } else {
                const T* qsrc = reinterpret_cast<const T*>(qslot);
                for (int e = lane; e < G * D; e += 32) qf[e] = qok ? static_cast<float>(qsrc[e]) * p.scale_log2 : 0.f;
            }
            __syncwarp();
            if (lane == 0 && qok) mbar_arrive(qempty_bar(qs));  // after an abort the slot stays held
            st.reset();
            const int len = lens_s[b];
            const int ntile = j1 - j0;
            if constexpr (MMA) {
                // Two 16-token steps per softmax update: the two 16-token tiles of a stage, or the two
                // halves of a 32-token tile.
                for (int i = 0; i < ntile; i += L::TPS) {
                    const uint32_t kk = k + i / L::TPS;
                    if (L::NC > 1 && (int)(kk % L::NC) != cw) continue;  // another consumer's stage
                    const int sidx = kk % S;
                    bool ok = L::NC == 1 || ticket_wait(misc + 1, (int32_t)kk, misc, p.status, p.wait_limit_ns);
                    ok = role_wait(full_bar(sidx), (kk / S) & 1, misc, p.status, p.wait_limit_ns) && ok;
                    if (L::NC > 1) {
                        __syncwarp();
                        if (lane == 0) misc[1] = (int32_t)kk + 1;  // taken (or given up): the next may go
                    }
                    if (ok) {
                        const uint32_t kb = base_s + L::kStagesOff + sidx * L::kStageBytes;
                        const uint32_t vb = kb + L::TPS * L::kTileBytes;
                        const int tok0 = (j0 + i) * BS;
                        // a second 16-token step: the tile's second half (32-token tiles), or the
                        // stage's second tile, which exists only if the piece holds one more tile
                        // (a piece may end before its sequence does)
                        const int v0 = min(16, len - tok0), v1 = min(16, len - tok0 - 16);
                        if (BS == 32 ? v1 > 0 : i + 1 < ntile) {
                            if (BS == 32)
                                st.step2(kb, vb, 0, v0, kb, vb, 16, v1, p.scale_log2, lane);
                            else
                                st.step2(kb, vb, 0, v0, kb + L::kTileBytes, vb + L::kTileBytes, 0, v1, p.scale_log2, lane);
                        } else {
                            st.step(kb, vb, 0, v0, p.scale_log2, lane);
                        }
                    }
                    __syncwarp();
                    if (lane == 0 && ok) mbar_arrive(empty_bar(sidx));  // after an abort the stage stays held
                }
                k += (ntile + L::TPS - 1) / L::TPS;
                if constexpr (L::NC > 1) {
                    // consumer 0 folds in the others' states (in warp order: the same bits every call)
                    if (cw > 0) st.save(comb + (cw - 1) * L::kCombFloats, lane);
                    named_barrier(1, 32 * L::NC);
                    if (cw == 0)
#pragma unroll
                        for (int w = 1; w < L::NC; ++w) st.combine(comb + (w - 1) * L::kCombFloats, lane);
                    named_barrier(1, 32 * L::NC);  // the hand-over area is free again
                    if (cw > 0) {
                        ++pi;
                        continue;  // consumer 0 finishes the piece
                    }
                }
            } else {
                for (int i = 0; i < ntile; ++i) {
                    const uint32_t kk = k + i;
                    const int sidx = kk % S;
                    const bool ok = role_wait(full_bar(sidx), (kk / S) & 1, misc, p.status, p.wait_limit_ns);
                    if (ok) {
                        const uint32_t kb = base_s + L::kStagesOff + sidx * L::kStageBytes;
                        const uint32_t vb = kb + L::kTileBytes;
                        const int tok0 = (j0 + i) * BS;
#pragma unroll
                        for (int sub = 0; sub < BS / 16; ++sub) {
                            const int valid = min(16, len - (tok0 + sub * 16));
                            if (valid > 0) st.step(kb, vb, sub * 16, valid, G, qf, ptile, lane);
                        }
                    }
                    __syncwarp();
                    if (lane == 0 && ok) mbar_arrive(empty_bar(sidx));  // after an abort the stage stays held
                }
                k += ntile;
            }
            if constexpr (MMA) st.finish();
            const int nb = P.nblocks(b);
            T* orow = static_cast<T*>(p.out) + ((size_t)b * Hq + (size_t)h * G) * D;
            if (j0 == 0 && j1 == nb) {
                st.store_out(orow, G, lane, p.out_scale);
            } else {
                // Split segment: store the unnormalised partial and count it in.  A piece that
                // continues a segment starts this CTA's range (slot 0); a split segment's first
                // piece ends it (slot 1).  The segment's pieces come from CTAs ca .. ca + np - 1,
                // one each, and ca's counter is the segment's.  A release fence orders every
                // lane's partial stores (the warp barrier puts them before it) ahead of the count;
                // the CTA whose piece completes the count merges the segment, after an acquire
                // fence (every other piece is then visible), and resets the counter for the next
                // call: right away when more pieces follow and it has few pieces (one piece per
                // round trip, few registers next to the loop's), else after the range (four per
                // round trip).  With the merge kernel instead, the piece is only stored.
                float* slot = p.partials + (size_t)(2 * c + (j0 > 0 ? 0 : 1)) * slot_floats;
                st.store_partial(slot, G, lane);
                if (merge_here) {
                    const int64_t s0 = P.seg_start(b, h);
                    const int ca = P.cta_of_seg(s0, b, h);
                    const int np = P.cta_of_seg(s0 + nb - 1, b, h) - ca + 1;
                    __syncwarp();
                    int old = 0;
                    if (lane == 0) {
                        fence_acq_rel_gpu();
                        old = atomicAdd(p.merge_counts + ca, 1);
                        if (old == np - 1) fence_acq_rel_gpu();
                    }
                    if (__shfl_sync(0xffffffffu, old, 0) == np - 1) {
                        if (np <= kMergeNowPieces && !it.done()) {
                            merge_pieces<T, D, 1>(p.partials, slot_floats, orow, ca, np, G, lane, 32, p.out_scale);
                            if (lane == 0) p.merge_counts[ca] = 0;
                        } else if (lane == 0) {
                            int32_t* e = pend + (j0 > 0 ? 0 : 4);
                            e[0] = b, e[1] = h, e[2] = ca, e[3] = np;
                        }
                    }
                }
            }
            ++pi;
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < (IKM ? 2 : 0) && cw == 0; ++i) {
            const int32_t* e = pend + 4 * i;
            const int np = e[3];
            if (np == 0) continue;
            const int ca = e[2];
            T* orow = static_cast<T*>(p.out) + ((size_t)e[0] * Hq + (size_t)e[1] * G) * D;
            merge_pieces<T, D, 4>(p.partials, slot_floats, orow, ca, np, G, lane, 32, p.out_scale);
            if (lane == 0) p.merge_counts[ca] = 0;
        }
    }
    __syncthreads();
}

// The two builds of the decode kernel.  With the in-kernel merge the kernel takes the
// register budget of kMaxCtasPerSm two-warp CTAs on an SM, 128 per thread, so that the rare
// merge path inside the piece loop does not raise the allocation of the whole kernel; without
// it the compiler keeps its own choice (an explicit minimum of one CTA per SM would let it
// take up to 255).
template <typename T, int D, int BS, bool MMA, int GF, typename KV, int NC>
__global__ void __launch_bounds__(Layout<T, D, BS, MMA, GF, KV, NC>::kThreadsCta, Layout<T, D, BS, MMA, GF, KV, NC>::kMinCtas)
    decode_kernel_ikm(const DecodeParams p, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v) {
    decode_body<T, D, BS, MMA, GF, KV, true, NC>(p, tmap_k, tmap_v);
}
template <typename T, int D, int BS, bool MMA, int GF, typename KV, int NC>
__global__ void __launch_bounds__(Layout<T, D, BS, MMA, GF, KV, NC>::kThreadsCta)
    decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v) {
    decode_body<T, D, BS, MMA, GF, KV, false, NC>(p, tmap_k, tmap_v);
}

// ---------------------------------------------------------------------------
// The merge of split segments (flash-decoding's reduce)
// ---------------------------------------------------------------------------
// The launch's other mode of merging (p.merge_in_kernel = 0; see pa_api.cu for
// the choice).  Launched right after decode_kernel as its programmatic dependent: it builds
// the same plan from seq_lens while the decode streams, then waits for the
// decode grid to finish (its partials visible) and merges every split
// segment.  The decode CTAs never wait for each other and never count pieces:
// the reduce costs them nothing at their tails.
// A split segment is one with a CTA range boundary strictly inside it; the
// first such boundary c (the segment starts in CTA c - 1) names it once.  So
// the work items are the boundaries c = 1 .. C-1, each taken by a group of
// lps = min(32, G D / 16) lanes (several groups per warp for small G D).
template <typename T, int D, int BS>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const DecodeParams p) {
    extern __shared__ int32_t msm[];
    const int B = p.num_seqs, Hkv = p.num_kv_heads;
    const bool fixed = p.partition_tiles > 0;
    int32_t* pref = msm;
    int32_t* upref = pref + (B + 1);
    int32_t* lens_s = upref + (fixed ? B + 1 : 0);
    int32_t* wsum = lens_s + B;
    int32_t pw[kPlanPass];
    if (p.plan != nullptr) plan_words_load<kMergeThreads>(p, 0, pw);  // in bounds: the host checked its size
    if (plan_matches(p, BS))  // the decode launch used the same plan
        load_plan_arrays<kMergeThreads>(p, pw, pref, upref, lens_s);
    else
        scan_lengths<BS, kMergeThreads>(p, false, pref, upref, lens_s, wsum);
    __syncthreads();
    const Plan P = make_plan(p, pref, upref);
    const int lane = threadIdx.x & 31;
    const int G = p.group;
    const int lps = min(32, G * D / 16), spw = 32 / lps;  // lanes per group, groups per warp
    const int grp = lane / lps, sl = lane % lps;
    if (grp >= spw) return;  // lanes left over when lps does not divide 32
    const size_t slot_floats = partial_slot_floats(G, D);
    const int ngroups = gridDim.x * (kMergeThreads / 32) * spw;
    // The segment boundary c names, if any: its sequence, KV head, first CTA and pieces.
    auto named = [&](int c, int& b, int& h, int& ca, int& np) -> bool {
        int64_t split;
        int seq;
        const int64_t t = P.cta_start(c, &split, &seq);
        if (t >= P.T) return false;
        b = P.find_seq(P.pref, t);
        const int nb = P.nblocks(b);
        const int64_t local = t - (int64_t)Hkv * P.pref[b];
        h = (int)(local / nb);
        const int j = (int)(local - (int64_t)h * nb);
        if (j == 0) return false;  // the boundary falls between segments
        const int64_t s0 = t - j;
        ca = P.cta_of_seg(s0, b, h);
        if (ca != c - 1) return false;  // an earlier boundary of this segment names it
        np = P.cta_of_seg(s0 + nb - 1, b, h) - ca + 1;
        return true;
    };
    int c = 1 + (blockIdx.x * (kMergeThreads / 32) + (threadIdx.x >> 5)) * spw + grp;
    int b = 0, h = 0, ca = 0, np = 0;
    bool have = c < P.C && named(c, b, h, ca, np);  // the first item is found while the decode runs
    // A dry run of the merge loop while the decode streams, over the zeroed status head and merge
    // counters (no store): its instructions are then in this SM's caches when the grid ends.
    if (have)
        merge_pieces<T, D, 4, false>(reinterpret_cast<const float*>(p.merge_counts), 0, nullptr, 0, 1, 1, sl, lps, 1.f);
    pdl_wait_prerequisites();  // the decode grid has finished; its partials are in memory
    while (c < P.C) {
        if (have) {
            T* orow = static_cast<T*>(p.out) + ((size_t)b * p.num_q_heads + (size_t)h * G) * D;
            merge_pieces<T, D, 4>(p.partials, slot_floats, orow, ca, np, G, sl, lps, p.out_scale);
        }
        c += ngroups;
        have = c < P.C && named(c, b, h, ca, np);
    }
}

// Host-side handle of one instantiation: two builds.
//  - `in`: with the in-kernel merge, one consumer warp (bf16 and FP8 pools; fp32 pools, a
//    reference-precision path whose loop leaves no registers to spare, have none).
//  - `mk`: for launches that merge with merge_kernel.  On the tensor-core path the in-kernel
//    merge's code costs the loop even when unused, so this build leaves it out; over FP8 pools,
//    whose consumer is the bound, it has three consumer warps.  Elsewhere it is `in`.
template <typename T, int D, int BS, bool MMA, int GF, typename KV = T>
struct VariantOf {
    static constexpr bool kIkm = !std::is_same<T, float>::value;
    static constexpr bool kOwnMk = kIkm && MMA;
    static constexpr int kNcMk = MMA && sizeof(KV) == 1 ? 3 : 1;
    using LIn = Layout<T, D, BS, MMA, GF, KV, 1>;
    using LMk = Layout<T, D, BS, MMA, GF, KV, kOwnMk ? kNcMk : 1>;
    using KernelFn = void (*)(const DecodeParams, const CUtensorMap, const CUtensorMap);
    static constexpr KernelFn in_kernel() {
        if constexpr (kIkm) return &decode_kernel_ikm<T, D, BS, MMA, GF, KV, 1>;
        else return &decode_kernel<T, D, BS, MMA, GF, KV, 1>;
    }
    static constexpr KernelFn mk_kernel() {
        if constexpr (kOwnMk) return &decode_kernel<T, D, BS, MMA, GF, KV, kNcMk>;
        else return in_kernel();
    }
    static int smem_in(int num_seqs, bool fixed) { return LIn::bytes(num_seqs, fixed); }
    static int smem_mk(int num_seqs, bool fixed) { return LMk::bytes(num_seqs, fixed); }
    // Both kernels are launched as programmatic dependents of what precedes them
    // on the stream: the decode of the preceding kernel (which may allow an early
    // start), the merge kernel (when the launch merges with it) of the decode.
    static void launch(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int grid, int smem,
                       int merge_grid, int merge_smem, cudaStream_t stream) {
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(p.merge_in_kernel ? LIn::kThreadsCta : LMk::kThreadsCta);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, p.merge_in_kernel ? in_kernel() : mk_kernel(), p, tk, tv) != cudaSuccess) return;
        if (p.merge_in_kernel) return;
        cudaLaunchConfig_t mcfg = cfg;
        mcfg.gridDim = dim3(merge_grid);
        mcfg.blockDim = dim3(kMergeThreads);
        mcfg.dynamicSmemBytes = merge_smem;
        cudaLaunchKernelEx(&mcfg, merge_kernel<T, D, BS>, p);
    }
    static DecodeVariant get() {
        return DecodeVariant{DecodeBuild{reinterpret_cast<const void*>(in_kernel()), LIn::S, LIn::kThreadsCta, &smem_in},
                             DecodeBuild{reinterpret_cast<const void*>(mk_kernel()), LMk::S, LMk::kThreadsCta, &smem_mk},
                             reinterpret_cast<const void*>(&merge_kernel<T, D, BS>), kIkm, &launch};
    }
};

}  // namespace pa
