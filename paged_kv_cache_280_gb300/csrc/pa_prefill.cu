// Paged prefill (chunked causal) attention for sm_103a, bf16, on the
// fifth-generation tensor cores.
//
// What it computes ("Q32: vLLM PagedAttention 原理" follow-up 3: FlashAttention
// loads the KV cache block by block, its block loading adapted to
// non-contiguous storage; data.6616ai.com "把虚拟内存搬进 KV Cache": attention
// reads KV by block index): sequence b holds seq_lens[b] tokens in the paged
// pool, the last n_b = cu_q_lens[b+1] - cu_q_lens[b] of them are a chunk
// whose queries are given, and chunk token i (position p = seq_lens[b] - n_b
// + i) attends to the keys at positions 0..p:  out = softmax(scale q K^T) V.
//
// Work decomposition.  For one (sequence, KV head) the G query heads of each
// chunk token are stacked into rows (token-major); a tile is 128 rows
// (128 / G chunk tokens): the M of every MMA, one row per TMEM lane.  A work
// unit is two consecutive tiles of one (sequence, KV head), which share every
// K/V stage of 128 keys.  The grid is persistent (one CTA per SM) and walks
// the units from the latest tiles (the most keys) to the earliest.
//
// CTA: twelve warps (eleven at work, the last only completes a warpgroup).
//   - Query loads (warp 10): per unit, both tiles' query rows by TMA (a 3-D
//     box of 64 elements x G heads x 128 / G tokens), once the previous unit's
//     Q K^T have completed.
//   - K/V producer (warp 8): per stage K and V, each into its own slot of a
//     5-slot ring (one box of BS rows x 128 bytes per block and 64-element
//     panel, 128-byte swizzle, evict-last L2 policy: the segment's other units
//     read the same blocks).  A block past the unit's last one is loaded from
//     past the pool's end, which TMA fills with zeros.  Without the query rows
//     to wait for, it runs ahead into the next unit as far as the ring allows.
//   - MMA (warp 9, one thread): S_t = Q_t K^T into tile t's TMEM (M 128, N 128,
//     K = head_dim, both operands K-major in shared memory), and O_t += P_t V
//     with P_t read from TMEM, where the softmax wrote it over S_t, and V an
//     MN-major operand.  Per stage it issues tile 0's P V and next S, then tile
//     1's, so the tensor core works on one tile while the other's softmax runs.
//     The tensor core performs one CTA's MMAs in issue order, so the S that
//     overwrites P is issued right after the P V that reads it.
//   - Softmax (warps 4t .. 4t + 3 for tile t, one thread per query row): reads
//     its S row from TMEM, applies the causal mask, keeps the row's running
//     max and sum with the scale folded into one fma per weight (base 2),
//     writes its row of P (bf16) back to TMEM, and, when the row max has grown
//     by more than 2^8 since O was last scaled, rescales its O row in TMEM
//     (the weights stay <= 256; the final ratio is exact).  The final O / l is
//     written from TMEM.  When a unit's last block is the sequence's partial
//     last block, the last tile's warps zero the V rows past the context's
//     end: they may hold any bits, and zero weight times NaN is NaN.
// Causal trimming: tile 0 skips a last stage that only tile 1 reaches, and on a
// tile's last stage the softmax forms weights only up to the last key the
// tile's last row sees (rounded up to 32 keys) and writes zeros past it.
// Every wait is bounded; a timeout sets PA_DEV_WAIT_TIMEOUT, every role stops,
// and the CTA waits for its own copies and MMAs before freeing TMEM.
#include <cmath>
#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int kPfTiles = 2;         // query tiles per work unit
constexpr int kPfSoftmaxWarps = 4;  // per tile
constexpr int kPfProducer = 8;      // warp index
constexpr int kPfMma = 9;           // warp index
constexpr int kPfQWarp = 10;        // warp index: query-row loads
constexpr int kPfThreads = 384;  // warp 11 completes the third warpgroup and only gives up registers
constexpr int kPfRows = 128;        // query rows per tile = MMA M = TMEM lanes
constexpr int kPfKeys = 128;        // keys per stage: N of S, K of P V
constexpr uint32_t kPfTmemCols = 512;  // tile t: S (P over its first 64 columns) in 256 t + [0, 128), O in 256 t + 128 + [0, D)
constexpr uint32_t kPfTmemTile = 256;
constexpr uint32_t kPfTmemO = 128;
constexpr float kPfRescaleLog2 = 8.f;  // rescale O only when a row max grows by more than this (log2)

// f(std::integral_constant<int, i>) for i = 0 .. N - 1, unrolled at compile time.
template <int I = 0, int N, class F>
__device__ __forceinline__ void static_for_impl(F& f) {
    if constexpr (I < N) {
        f(std::integral_constant<int, I>{});
        static_for_impl<I + 1, N>(f);
    }
}
template <int N, class F>
__device__ __forceinline__ void static_for(F&& f) {
    static_for_impl<0, N>(f);
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 2^x on the SFU (ex2.approx: a few ulp, well inside the bf16 output bound); 2^-inf = +0.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Shared memory of one CTA (1024-byte aligned regions, 128-byte swizzle):
//   Q[t]     [D / 64 panels][128 rows][128 B]
//   slot[i]  K or V of one stage: [D / 64 panels][128 keys][128 B]
template <int D, int BS>
struct PfLayout {
    static constexpr int kPanels = D / 64;
    static constexpr int kQPanel = kPfRows * 128;
    static constexpr int kQBytes = kPanels * kQPanel;
    static constexpr int kSlotPanel = kPfKeys * 128;
    static constexpr int kSlotBytes = kPanels * kSlotPanel;
    static constexpr int kSlots = D == 128 ? 5 : 8;
    static constexpr int kBlocksPerStage = kPfKeys / BS;
    static constexpr int kQOff = 0;
    static constexpr int kRingOff = kPfTiles * kQBytes;
    static constexpr int kBarOff = kRingOff + kSlots * kSlotBytes;
    static constexpr int kNumBars = 2 * kSlots + 3 * kPfTiles + 3;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // abort flag, TMEM address
    static constexpr int kBytes = kMiscOff + 64 + 1024;      // +1 KB to align the base
    static_assert(kQPanel % 1024 == 0 && kSlotPanel % 1024 == 0, "1024-byte alignment");
    static_assert(kBytes <= 227 * 1024, "shared memory");
};

template <int NS>
struct PfBars {
    uint32_t base;
    __device__ uint32_t at(int i) const { return base + 8u * i; }
    __device__ uint32_t slot_full(int s) const { return at(s); }
    __device__ uint32_t slot_empty(int s) const { return at(NS + s); }
    __device__ uint32_t s_full(int t) const { return at(2 * NS + t); }    // S_t in TMEM
    __device__ uint32_t p_ready(int t) const { return at(2 * NS + kPfTiles + t); }  // P_t in TMEM, O_t rescaled
    __device__ uint32_t o_final(int t) const { return at(2 * NS + 2 * kPfTiles + t); }  // a unit's last P V
    __device__ uint32_t q_full() const { return at(2 * NS + 3 * kPfTiles); }
    __device__ uint32_t q_empty() const { return at(2 * NS + 3 * kPfTiles + 1); }
    __device__ uint32_t mma_drain() const { return at(2 * NS + 3 * kPfTiles + 2); }
};

// Warp-collective bounded wait (every lane calls it); gives up once the CTA's abort flag is set.
__device__ __forceinline__ bool pf_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag, int32_t* status) {
    if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
    bool ok = mbar_wait(bar, parity, kWaitLimitNs, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
        *abort_flag = 1;
        if ((threadIdx.x & 31) == 0) flag_status(status, PA_DEV_WAIT_TIMEOUT);
    }
    return ok;
}

// The same for one thread (the MMA issuer).
__device__ __forceinline__ bool pf_wait1(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag, int32_t* status) {
    if (*abort_flag) return false;
    if (mbar_wait(bar, parity, kWaitLimitNs, abort_flag)) return true;
    *abort_flag = 1;
    flag_status(status, PA_DEV_WAIT_TIMEOUT);
    return false;
}

// One work unit: tiles 2m and 2m + 1 of (sequence b, KV head g).  Every role
// walks the same units in the same order and derives the same fields.
struct PfUnit {
    int b, g, c0, n, len;
    int i0[kPfTiles], i1[kPfTiles];
    int ntiles;      // 1 or 2 (the chunk's last unit may hold one tile)
    int nkeys;       // keys up to the unit's last position
    int nst;         // 128-key stages (those of the last tile)
    int nst0;        // stages of tile 0 (nst, or nst - 1 when tile 1 reaches into one more)
    int kend0, kend1;  // keys visible to the last row of tile 0 / tile 1 (positions 0 .. kend - 1)
    int nblk;        // blocks
    bool zero_tail;  // the unit's last block is the sequence's partial last block
};

// Columns of a tile's S at stage k that its last row can see (keys below kend), rounded up to 32
// (one TMEM load of the softmax), at most a whole stage.  Positive while k < the tile's stages.
__device__ __forceinline__ int pf_cols(int kend, int k) {
    const int nv = kend - k * kPfKeys;
    return nv >= kPfKeys ? kPfKeys : ((nv + 31) & ~31);
}

// 0: empty unit (skipped by every role); 1: a unit to compute; -1: a malformed
// sequence (flagged once, skipped).
template <int BS>
__device__ __forceinline__ int pf_unit(const PrefillParams& p, int u, int pairs, PfUnit& w) {
    const int bh = p.num_seqs * p.num_kv_heads;
    const int m = pairs - 1 - u / bh, rem = u - (u / bh) * bh;
    w.b = rem / p.num_kv_heads;
    w.g = rem - w.b * p.num_kv_heads;
    w.c0 = __ldg(p.cu_q_lens + w.b);
    w.n = __ldg(p.cu_q_lens + w.b + 1) - w.c0;
    w.len = __ldg(p.seq_lens + w.b);
    const int tt = p.tile_tokens;
    w.i0[0] = 2 * m * tt;
    if (w.n <= 0 || w.i0[0] >= w.n) return 0;
    if (w.n > w.len || w.n > p.max_q_len || (int64_t)w.len > (int64_t)p.max_blocks_per_seq * BS || w.c0 < 0 ||
        (int64_t)w.c0 + w.n > p.num_q_tokens)
        return -1;
    w.i1[0] = min(w.n, w.i0[0] + tt);
    w.i0[1] = w.i0[0] + tt;
    w.i1[1] = min(w.n, w.i0[1] + tt);
    w.ntiles = w.i0[1] < w.n ? 2 : 1;
    w.nkeys = w.len - w.n + (w.ntiles == 2 ? w.i1[1] : w.i1[0]);
    w.nst = (w.nkeys + kPfKeys - 1) / kPfKeys;
    w.kend0 = w.len - w.n + w.i1[0];
    w.kend1 = w.nkeys;
    w.nst0 = (w.kend0 + kPfKeys - 1) / kPfKeys;
    w.nblk = (w.nkeys + BS - 1) / BS;
    // Past the context's end the block's slots may hold any bits.  This holds for the unit that ends
    // at the last token, and also for one that ends fewer than BS tokens before it.
    w.zero_tail = (int64_t)w.nblk * BS > w.len;
    return 1;
}

// K/V producer warp: per unit, K(0), V(0), K(1), V(1), ... through the slot ring.  The query
// rows are loaded by a warp of their own, so this one never waits for a unit's Q K^T to complete
// and runs ahead into the next unit as far as the ring allows.
template <int D, int BS>
__device__ __forceinline__ void pf_produce(const PrefillParams& p, const CUtensorMap* tk, const CUtensorMap* tv,
                                           int pairs, int total, uint32_t base_s,
                                           const PfBars<PfLayout<D, BS>::kSlots>& bars, volatile int32_t* abort_flag,
                                           int lane) {
    using L = PfLayout<D, BS>;
    constexpr int BPS = L::kBlocksPerStage, NS = L::kSlots;
    if (lane == 0) {
        prefetch_tensormap(tk);
        prefetch_tensormap(tv);
    }
    const uint64_t policy = policy_evict_last();
    const int32_t oob_row = p.num_blocks * p.num_kv_heads * BS;  // past the pool: TMA reads zeros
    int sc = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < total; u += gridDim.x) {
        PfUnit w;
        const int kind = pf_unit<BS>(p, u, pairs, w);
        if (kind < 0 && lane == 0 && w.g == 0) flag_status(p.status, PA_DEV_BAD_SEQ_LEN);
        if (kind <= 0) continue;
        const int32_t* tab = p.block_tables + (size_t)w.b * p.max_blocks_per_seq;
        int32_t blk = 0;
        for (int k = 0; ok && k < w.nst; ++k) {
            const int jb0 = k * BPS;
            if ((jb0 & 31) == 0) blk = jb0 + lane < w.nblk ? __ldg(tab + jb0 + lane) : 0;  // 32 entries at a time
            int32_t rows[BPS];
#pragma unroll
            for (int t = 0; t < BPS; ++t) {
                int32_t bid = __shfl_sync(0xffffffffu, blk, (jb0 + t) & 31);
                if (jb0 + t >= w.nblk) {
                    rows[t] = oob_row;
                } else {
                    if (bid < 0 || bid >= p.num_blocks) {  // warp-uniform
                        if (lane == 0) flag_status(p.status, PA_DEV_BAD_BLOCK_ID);
                        bid = 0;
                    }
                    rows[t] = (bid * p.num_kv_heads + w.g) * BS;
                }
            }
#pragma unroll
            for (int half = 0; half < 2; ++half, ++sc) {  // K, then V
                const int s = sc % NS;
                if (!pf_wait(bars.slot_empty(s), ((sc / NS) & 1) ^ 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                // one lane per block issues that block's boxes, so the copies are requested in parallel
                if (lane == 0) mbar_arrive_expect_tx(bars.slot_full(s), (uint32_t)L::kSlotBytes);
                __syncwarp();
                if (lane < BPS) {
                    const uint32_t dst = base_s + L::kRingOff + s * L::kSlotBytes + lane * BS * 128;
                    const CUtensorMap* map = half ? tv : tk;
                    int32_t row = rows[0];
#pragma unroll
                    for (int t = 1; t < BPS; ++t)
                        if (lane == t) row = rows[t];
#pragma unroll
                    for (int pn = 0; pn < L::kPanels; ++pn)
                        tma_load_2d(dst + pn * L::kSlotPanel, map, pn * 64, row, bars.slot_full(s), policy);
                }
            }
        }
    }
    // never leave the CTA with copies still landing in its shared memory (a slot's phase completes
    // only when its copies have landed)
    for (int kk = sc > NS ? sc - NS : 0; kk < sc; ++kk) mbar_wait(bars.slot_full(kk % NS), (kk / NS) & 1);
}

// Query warp: per unit, both tiles' query rows, once the previous unit's Q K^T have completed.  A
// warp of its own, so that the K/V producer never waits for that and runs ahead into the next unit.
template <int D, int BS>
__device__ __forceinline__ void pf_produce_q(const PrefillParams& p, const CUtensorMap* tq, int pairs, int total,
                                             uint32_t base_s, const PfBars<PfLayout<D, BS>::kSlots>& bars,
                                             volatile int32_t* abort_flag, int lane) {
    using L = PfLayout<D, BS>;
    if (lane == 0) prefetch_tensormap(tq);
    const int G = p.group;
    const uint32_t q_tile_bytes = (uint32_t)(L::kPanels * G * p.tile_tokens * 128);
    int uc = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
        PfUnit w;
        if (pf_unit<BS>(p, u, pairs, w) <= 0) continue;
        if (!pf_wait(bars.q_empty(), (uc & 1) ^ 1, abort_flag, p.status)) break;
        if (lane == 0) {
            mbar_arrive_expect_tx(bars.q_full(), q_tile_bytes * w.ntiles);
#pragma unroll
            for (int t = 0; t < kPfTiles; ++t)
                if (t < w.ntiles)
#pragma unroll
                    for (int pn = 0; pn < L::kPanels; ++pn)
                        tma_load_3d(base_s + L::kQOff + t * L::kQBytes + pn * L::kQPanel, tq, pn * 64, w.g * G,
                                    w.c0 + w.i0[t], bars.q_full());
        }
        ++uc;
    }
    if (uc > 0) mbar_wait(bars.q_full(), (uc - 1) & 1);  // the last box has landed
}

// MMA issuer (one thread).
template <int D, int BS>
__device__ __forceinline__ void pf_mma(const PrefillParams& p, int pairs, int total, uint32_t base_s, uint32_t tmem,
                                       const PfBars<PfLayout<D, BS>::kSlots>& bars, volatile int32_t* abort_flag) {
    using L = PfLayout<D, BS>;
    constexpr int NS = L::kSlots;
    constexpr uint32_t idesc_s = umma_idesc_bf16(kPfRows, kPfKeys, 0, 0);  // Q (K-major) x K^T (K-major)
    constexpr uint32_t idesc_o = umma_idesc_bf16(kPfRows, D, 0, 1);  // P (TMEM) x V (MN-major)
    int sc = 0, uc = 0, ck0 = 0, ck1 = 0;  // slots; units; stages of tile 0 and of tile 1
    bool ok = true;
    // Descriptors: the upper word is a constant per operand kind; the lower word holds the start
    // address / 16 (bits 0..13, below 256 KB: never carries into the leading offset) and the
    // leading byte offset, so an operand at a byte offset adds offset / 16 to the lower word.
    const uint32_t q_lo = (uint32_t)umma_smem_desc(base_s + L::kQOff, 16, 1024);     // K-major Q, tile 0
    const uint32_t k_lo = (uint32_t)umma_smem_desc(base_s + L::kRingOff, 16, 1024);  // K-major K, slot 0
    const uint32_t v_lo = (uint32_t)umma_smem_desc(base_s + L::kRingOff, L::kSlotPanel, 1024);  // MN-major V
    constexpr uint32_t hi = (uint32_t)(umma_smem_desc(0, 0, 1024) >> 32);  // SBO 1024, version, swizzle
    // S_t = Q_t K^T
    auto issue_s = [&](int t, int ks_slot) {
        const uint32_t qa = q_lo + (uint32_t)(t * (L::kQBytes >> 4));
        const uint32_t kb = k_lo + (uint32_t)(ks_slot * (L::kSlotBytes >> 4));
        const uint32_t d = tmem + kPfTmemTile * t;
        // K steps of 16 elements: 32 bytes along a 128-byte row, 64-element panels further apart
        auto step = [&](auto ks_c) {
            constexpr int ks = decltype(ks_c)::value;
            constexpr uint32_t oa = ((ks >> 2) * L::kQPanel + (ks & 3) * 32) >> 4;
            constexpr uint32_t ob = ((ks >> 2) * L::kSlotPanel + (ks & 3) * 32) >> 4;
            umma_bf16_lo<oa, ob>(d, qa, kb, hi, idesc_s, ks > 0 ? 1u : 0u);
        };
        static_for<D / 16>(step);
        umma_commit(bars.s_full(t));
    };
    // O_t += P_t V over the stage's 128 keys (8 steps of K = 16).  A tile's last stage could stop
    // after the keys its last row sees, but on GB300 that measured slower than the full stage (the
    // softmax writes zero weights past them instead).
    auto issue_o = [&](int t, int vs_slot, bool first) {
        const uint32_t vb = v_lo + (uint32_t)(vs_slot * (L::kSlotBytes >> 4));
        const uint32_t d = tmem + kPfTmemTile * t;
        const uint32_t acc0 = first ? 0u : 1u;
        auto step = [&](auto kk_c) {
            constexpr int kk = decltype(kk_c)::value;
            constexpr uint32_t ob = (kk * 16 * 128) >> 4;  // 16 keys = 16 rows of 128 bytes of every panel
            umma_bf16_tmem_a_lo<ob>(d + kPfTmemO, d + kk * 8, vb, hi, idesc_o, kk > 0 ? 1u : acc0);
        };
        static_for<kPfKeys / 16>(step);
    };
    for (int u = blockIdx.x; ok && u < total; u += gridDim.x) {
        PfUnit w;
        if (pf_unit<BS>(p, u, pairs, w) <= 0) continue;
        const int T = w.ntiles;
        // S_t(0) for every tile of the unit
        const int k0 = sc++;
        ok = pf_wait1(bars.q_full(), uc & 1, abort_flag, p.status) &&
             pf_wait1(bars.slot_full(k0 % NS), (k0 / NS) & 1, abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
        for (int t = 0; t < T; ++t) issue_s(t, k0 % NS);
        umma_commit(bars.slot_empty(k0 % NS));
        if (w.nst == 1) umma_commit(bars.q_empty());  // the unit's last Q K^T
        for (int k = 0; k < w.nst; ++k) {
            const bool last = k + 1 == w.nst;
            const int vs = sc++;
            const int ks1 = last ? -1 : sc++;
            if (!pf_wait1(bars.slot_full(vs % NS), (vs / NS) & 1, abort_flag, p.status)) {
                ok = false;
                break;
            }
            // tile 0 may have one stage fewer than the unit (its last row sees fewer keys)
            const bool skip0 = k >= w.nst0;
            // On the unit's last stage the last tile's warps may zero V rows: every tile waits for them.
            const bool all = last && w.zero_tail;
            for (int t = 0; ok && all && t < T; ++t)
                if (t > 0 || !skip0) ok = pf_wait1(bars.p_ready(t), (t ? ck1 : ck0) & 1, abort_flag, p.status);
            bool k_ready = false;
            for (int t = 0; ok && t < T; ++t) {
                if (t == 0 && skip0) continue;
                int& ck = t ? ck1 : ck0;
                const int nst_t = t ? w.nst : w.nst0;
                if (!all && !pf_wait1(bars.p_ready(t), ck & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_o(t, vs % NS, k == 0);
                if (k + 1 == nst_t) {
                    umma_commit(bars.o_final(t));
                } else {
                    if (!k_ready && !pf_wait1(bars.slot_full(ks1 % NS), (ks1 / NS) & 1, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    k_ready = true;
                    issue_s(t, ks1 % NS);
                }
                ++ck;
            }
            if (!ok) break;
            umma_commit(bars.slot_empty(vs % NS));  // V(k) may be refilled once both P V complete
            if (!last) {
                umma_commit(bars.slot_empty(ks1 % NS));
                if (k + 2 == w.nst) umma_commit(bars.q_empty());  // the unit's last Q K^T were just issued
            }
        }
        ++uc;
    }
    // every MMA issued has completed before the CTA may free TMEM or its shared memory
    umma_commit(bars.mma_drain());
    mbar_wait(bars.mma_drain(), 0);
}

// Softmax warps of tile t: query row r = 32 (warp % 4) + lane, TMEM lane r.
template <int D, int BS>
__device__ __forceinline__ void pf_softmax(const PrefillParams& p, int pairs, int total, int t, uint8_t* base,
                                           uint32_t tmem, const PfBars<PfLayout<D, BS>::kSlots>& bars,
                                           volatile int32_t* abort_flag, int warp, int lane) {
    using L = PfLayout<D, BS>;
    constexpr int NS = L::kSlots;
    const int G = p.group, Hq = p.num_q_heads;
    const int rows_used = p.tile_tokens * G;
    const int r = 32 * (warp & 3) + lane;
    const uint32_t row_tmem = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + kPfTmemTile * t;
    const float c = p.scale_log2;  // > 0 (checked on the host)
    int sc = 0, ck = 0, uc = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
        PfUnit w;
        if (pf_unit<BS>(p, u, pairs, w) <= 0) continue;
        const int sc0 = sc;
        sc += 2 * w.nst;
        if (t >= w.ntiles) continue;
        const int i0 = t ? w.i0[1] : w.i0[0], i1 = t ? w.i1[1] : w.i1[0];
        const int tok = i0 + r / G;
        const bool valid = r < rows_used && tok < i1;
        // padding rows take the tile's last position: their scores stay finite and they are never stored
        const int pos = w.len - w.n + (valid ? tok : i1 - 1);
        float m_raw = -INFINITY, l_run = 0.f;  // running max of the raw scores (the scale is > 0), and sum
        const int kend = t ? w.kend1 : w.kend0, nst_t = t ? w.nst : w.nst0;
        for (int k = 0; k < nst_t; ++k, ++ck) {
            if (!pf_wait(bars.s_full(t), ck & 1, abort_flag, p.status)) return;
            tc_fence_after();
            // S_t(k) was issued after P_t(k-1) V(k-1) and completes after it: O is up to date and
            // no MMA touches this tile's TMEM until this warp arrives on p_ready.
            // the stage's 128 scores of this row, one TMEM round trip; causal mask: key j is visible
            // to the row at position pos iff j <= pos (masked scores become -inf, so weigh 0 below).
            // Only the first nq x 32 columns can hold a key that some row of the tile sees.
            const int key0 = k * kPfKeys, nq = pf_cols(kend, k) >> 5;
            uint32_t sv[4][32];
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_ld32(row_tmem + 32 * q, sv[q]);
            tmem_wait_ld();
            if (key0 + kPfKeys - 1 > pos) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (key0 + 32 * q + e > pos) sv[q][e] = __float_as_uint(-INFINITY);
            }
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    mx0 = fmax3(mx0, __uint_as_float(sv[q][e]), __uint_as_float(sv[q][e + 1]));
                    mx1 = fmax3(mx1, __uint_as_float(sv[q][e + 2]), __uint_as_float(sv[q][e + 3]));
                }
            const float mx = fmaxf(mx0, mx1);
            const float m_new = fmaxf(m_raw, mx);  // finite: stage 0 holds key 0, which every row sees
            if (k == 0) {
                m_raw = m_new;
            } else {
                const bool need = (m_new - m_raw) * c > kPfRescaleLog2;
                if (__any_sync(0xffffffffu, need)) {
                    const float f = need ? fast_exp2((m_raw - m_new) * c) : 1.f;
#pragma unroll
                    for (int c0o = 0; c0o < D; c0o += 32) {
                        uint32_t ov[32];
                        tmem_ld32(row_tmem + kPfTmemO + c0o, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
                        tmem_st32(row_tmem + kPfTmemO + c0o, ov);
                    }
                    if (need) {
                        l_run *= f;
                        m_raw = m_new;
                    }
                }
            }
            // P = 2^(c s - c m) as bf16 pairs over the first 64 columns of S (its scores are in registers)
            // (packed pairs: one fma.f32x2 forms two exponents, one add.f32x2 adds two weights)
            const float mc = m_raw * c;
            const uint64_t c2 = f2_pack(c, c), nmc2 = f2_pack(-mc, -mc);
            uint64_t sum2 = f2_pack(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (q >= nq) {  // past the tile's last position: zero weights, no exponentials
                    const uint32_t z[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                    tmem_st16(row_tmem + 16 * q, z);
                    continue;
                }
                uint32_t pw[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float x0, x1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[q][2 * e]), __uint_as_float(sv[q][2 * e + 1])), c2, nmc2),
                              x0, x1);
                    x0 = fast_exp2(x0);
                    x1 = fast_exp2(x1);
                    sum2 = f2_add(sum2, f2_pack(x0, x1));
                    pw[e] = pack_bf16x2(x0, x1);
                }
                tmem_st16(row_tmem + 16 * q, pw);
            }
            float sa, sb;
            f2_unpack(sum2, sa, sb);
            const float sum = sa + sb;
            l_run += sum;
            // The unit's last block is the sequence's partial last block: its slots past the context's
            // end may hold any bits; zero their V rows before any P V reads the stage.
            if (k + 1 == nst_t && w.zero_tail && t == w.ntiles - 1) {
                const int vs = sc0 + 2 * k + 1, s = vs % NS;
                if (!pf_wait(bars.slot_full(s), (vs / NS) & 1, abort_flag, p.status)) return;
                uint8_t* vst = base + L::kRingOff + s * L::kSlotBytes;
                const int z0 = w.len - key0, z1 = w.nblk * BS - key0;  // rows [z0, z1) of the stage
                const int nz = (z1 - z0) * 8 * L::kPanels;              // 16-byte chunks
                for (int i = r; i < nz; i += kPfRows) {
                    const int pn = i / ((z1 - z0) * 8), rem = i - pn * ((z1 - z0) * 8);
                    *reinterpret_cast<uint4*>(vst + pn * L::kSlotPanel + (z0 + rem / 8) * 128 + (rem & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.p_ready(t));
        }
        // ---- O / l from TMEM to out (bf16) ----
        if (!pf_wait(bars.o_final(t), uc & 1, abort_flag, p.status)) return;
        ++uc;
        tc_fence_after();
        const float inv = 1.f / l_run;
        uint16_t* dst = static_cast<uint16_t*>(p.out) +
                        ((size_t)(w.c0 + (valid ? tok : i0)) * Hq + (size_t)w.g * G + r % G) * D;
        // the whole O row in one TMEM round trip, then its bf16 row in 32-byte stores (16-byte
        // stores when out is only 16-byte aligned)
        uint32_t ov[D / 32][32];
#pragma unroll
        for (int q = 0; q < D / 32; ++q) tmem_ld32(row_tmem + kPfTmemO + 32 * q, ov[q]);
        tmem_wait_ld();
        if (valid) {
            uint32_t wv[D / 2];
#pragma unroll
            for (int e = 0; e < D / 2; ++e)
                wv[e] = pack_bf16x2(__uint_as_float(ov[e >> 4][(2 * e) & 31]) * inv,
                                    __uint_as_float(ov[e >> 4][(2 * e + 1) & 31]) * inv);
            if (p.out_align32) {
#pragma unroll
                for (int v = 0; v < D / 16; ++v)
                    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + 16 * v),
                                 "r"(wv[8 * v]), "r"(wv[8 * v + 1]), "r"(wv[8 * v + 2]), "r"(wv[8 * v + 3]),
                                 "r"(wv[8 * v + 4]), "r"(wv[8 * v + 5]), "r"(wv[8 * v + 6]), "r"(wv[8 * v + 7])
                                 : "memory");
            } else {
#pragma unroll
                for (int v = 0; v < D / 8; ++v)
                    reinterpret_cast<uint4*>(dst)[v] = make_uint4(wv[4 * v], wv[4 * v + 1], wv[4 * v + 2], wv[4 * v + 3]);
            }
        }
        tc_fence_before();  // the O reads are ordered before this warp's next p_ready arrival
    }
}

template <int D, int BS>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_q) {
    using L = PfLayout<D, BS>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_s - raw_s);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tiles = (p.max_q_len + p.tile_tokens - 1) / p.tile_tokens;
    const int pairs = (tiles + 1) / 2;
    const int total = pairs * p.num_seqs * p.num_kv_heads;

    volatile int32_t* misc = reinterpret_cast<volatile int32_t*>(base + L::kMiscOff);
    PfBars<L::kSlots> bars{base_s + L::kBarOff};
    if (tid == 0) {
        for (int s = 0; s < L::kSlots; ++s) {
            mbar_init(bars.slot_full(s), 1);   // the producer's expect_tx
            mbar_init(bars.slot_empty(s), 1);  // tcgen05.commit after the slot's last MMA
        }
        for (int t = 0; t < kPfTiles; ++t) {
            mbar_init(bars.s_full(t), 1);                 // tcgen05.commit after Q K^T
            mbar_init(bars.p_ready(t), kPfSoftmaxWarps);  // each softmax warp has written its P rows
            mbar_init(bars.o_final(t), 1);
        }
        mbar_init(bars.q_full(), 1);
        mbar_init(bars.q_empty(), 1);
        mbar_init(bars.mma_drain(), 1);
        fence_barrier_init();
        misc[0] = 0;  // abort flag
    }
    if (warp == kPfMma) tmem_alloc(base_s + L::kMiscOff + 16, kPfTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(base + L::kMiscOff + 16);

    // Registers: the launch gives every thread 168 (384 x 168 = 64512); the producer / MMA warpgroup
    // keeps 56 and the two softmax warpgroups take 224 each: 2 x 128 x 224 + 128 x 56 = 64512.
    if (warp >= 8) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 56;" ::: "memory");
        if (warp == kPfProducer)
            pf_produce<D, BS>(p, &tmap_k, &tmap_v, pairs, total, base_s, bars, misc, lane);
        else if (warp == kPfQWarp)
            pf_produce_q<D, BS>(p, &tmap_q, pairs, total, base_s, bars, misc, lane);
        else if (warp == kPfMma) {
            if (lane == 0) pf_mma<D, BS>(p, pairs, total, base_s, tmem, bars, misc);
            __syncwarp();
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 224;" ::: "memory");
        pf_softmax<D, BS>(p, pairs, total, warp >> 2, base, tmem, bars, misc, warp, lane);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kPfMma) tmem_dealloc(tmem, kPfTmemCols);
}

template <int D, int BS>
pa_status launch_prefill(const PrefillParams& p, const void* k_pool, const void* v_pool, int64_t rows, int num_seqs,
                         int max_q_len, cudaStream_t stream) {
    using L = PfLayout<D, BS>;
    int dev = 0, occ = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return PA_ERR_CUDA;
    const void* kfn = reinterpret_cast<const void*>(&prefill_kernel<D, BS>);
    if (!kernel_occupancy(dev, kfn, kPfThreads, L::kBytes, &occ)) return PA_ERR_CUDA;
    if (occ <= 0) return PA_ERR_UNSUPPORTED;
    CUtensorMap tk, tv, tq;
    if (!pool_map(&tk, dev, k_pool, rows, D, BS, PA_BF16) || !pool_map(&tv, dev, v_pool, rows, D, BS, PA_BF16) ||
        !prefill_q_map(&tq, dev, p.q, p.num_q_tokens, p.num_q_heads, D, p.group, p.tile_tokens))
        return PA_ERR_CUDA;
    const int tiles = (max_q_len + p.tile_tokens - 1) / p.tile_tokens;
    const int64_t total = (int64_t)((tiles + 1) / 2) * num_seqs * p.num_kv_heads;
    if (total >= INT32_MAX) return PA_ERR_UNSUPPORTED;
    const int grid = (int)(total < (int64_t)sms ? total : sms);  // persistent: one CTA per SM
    prefill_kernel<D, BS><<<grid, kPfThreads, L::kBytes, stream>>>(p, tk, tv, tq);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" pa_status pa_prefill_attention(void* out, const void* q, const void* k_pool, const void* v_pool,
                                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                                          const int32_t* seq_lens, const int32_t* cu_q_lens, int32_t num_seqs,
                                          int32_t num_q_tokens, int32_t max_q_len, int32_t num_q_heads,
                                          int32_t num_kv_heads,
                                          int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale,
                                          pa_dtype dtype, int32_t* dev_status, void* stream) {
    if (dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads || max_q_len < 0 ||
        num_q_tokens < 0 ||
        max_blocks_per_seq <= 0 || num_blocks <= 0 || !std::isfinite(scale) || !(scale > 0.f))
        return PA_ERR_INVALID_ARG;
    if (num_q_heads / num_kv_heads > 8 || (head_dim != 64 && head_dim != 128) || (block_size != 16 && block_size != 32) ||
        num_seqs > 65535 || num_kv_heads > 65535)
        return PA_ERR_UNSUPPORTED;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !seq_lens || !cu_q_lens) return PA_ERR_INVALID_ARG;
    auto a16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
    auto a4 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) == 0; };
    if (!a16(out) || !a16(q) || !a16(k_pool) || !a16(v_pool) || !a4(block_tables) || !a4(seq_lens) || !a4(cu_q_lens) ||
        !a4(dev_status))
        return PA_ERR_INVALID_ARG;
    const int64_t rows = (int64_t)num_blocks * num_kv_heads * block_size;
    if (rows >= INT32_MAX) return PA_ERR_UNSUPPORTED;
    if (max_q_len == 0 || num_q_tokens == 0) return PA_OK;
    if ((int64_t)num_q_tokens * num_q_heads * head_dim >= INT32_MAX * 2ll) return PA_ERR_UNSUPPORTED;
    PrefillParams p;
    p.out = out;
    p.q = q;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.cu_q_lens = cu_q_lens;
    p.status = dev_status;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.num_blocks = num_blocks;
    p.group = num_q_heads / num_kv_heads;
    p.tile_tokens = kPfRows / p.group;
    p.num_q_tokens = num_q_tokens;
    p.max_q_len = max_q_len;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.out_align32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0 ? 1 : 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (head_dim == 128 && block_size == 16) return launch_prefill<128, 16>(p, k_pool, v_pool, rows, num_seqs, max_q_len, st);
    if (head_dim == 128 && block_size == 32) return launch_prefill<128, 32>(p, k_pool, v_pool, rows, num_seqs, max_q_len, st);
    if (head_dim == 64 && block_size == 16) return launch_prefill<64, 16>(p, k_pool, v_pool, rows, num_seqs, max_q_len, st);
    return launch_prefill<64, 32>(p, k_pool, v_pool, rows, num_seqs, max_q_len, st);
}
