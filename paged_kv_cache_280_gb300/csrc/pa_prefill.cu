// Paged prefill (chunked causal) attention for sm_103a, bf16.
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
// chunk token are stacked into rows (token-major), and a CTA takes a tile of
// 64 rows: 64 / G consecutive chunk tokens.  Those rows share every K/V tile
// of the segment, so the contraction is a real dense tile: S = Q K^T with the
// 64 rows as M, and O = P V.  Tiles that end later in the chunk see more keys;
// the grid hands them out first.
//
// CTA: four consumer warps (16 query rows each, Q held in registers as MMA
// A-fragments) and one producer warp that walks the block table 32 entries
// at a time and moves each (block, KV head) tile of K and V with TMA
// (cp.async.bulk.tensor, 128-byte swizzle, evict-last L2 policy: the other
// query tiles of the segment read the same blocks) into an S-stage ring
// guarded by full/empty mbarriers, 32 keys per stage.  Per stage a consumer
// warp runs 4 x D/16 mma.sync for S, one online-softmax step over its rows
// (running max and sum in the base-2 domain, the causal mask applied per
// element), and D/4 mma.sync for P V, with P passed from the S accumulators
// to A-fragments in registers.  Every wait is bounded; a timeout sets
// PA_DEV_WAIT_TIMEOUT.
#include <cmath>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kPfConsumers = 4;
constexpr int kPfProducer = kPfConsumers;  // warp index
constexpr int kPfThreads = 32 * (kPfConsumers + 1);
constexpr int kPfRows = 16 * kPfConsumers;  // query rows per CTA
constexpr int kPfKeys = 32;                 // keys per pipeline stage and per softmax step
constexpr int kPfRingBytes = 49152;
constexpr int kPfCtasPerSm = 2;

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 2^x on the SFU (ex2.approx: a few ulp, well inside the bf16 output bound);
// 2^-inf = +0.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// A stage holds 32 keys of one (sequence, KV head): K then V, each as 32 / BS
// pool tiles of BS rows (tile i = block 32k/BS + i of the segment).
template <int D, int BS>
struct PfLayout {
    static constexpr int kTileBytes = BS * D * 2;  // K (or V) of one (block, KV head)
    static constexpr int kTilesPerStage = kPfKeys / BS;
    static constexpr int kHalfBytes = kTilesPerStage * kTileBytes;  // the stage's K (or V)
    static constexpr int kStageBytes = 2 * kHalfBytes;
    static constexpr int S = kPfRingBytes / kStageBytes < 2 ? 2 : kPfRingBytes / kStageBytes;
    static constexpr int kPanels = D * 2 / 128;
    static constexpr int kQOff = 0;  // [64 rows][D] bf16, 128-byte swizzle
    static constexpr int kQBytes = kPfRows * D * 2;
    static constexpr int kRingOff = kQOff + kQBytes;
    static constexpr int kBarOff = kRingOff + S * kStageBytes;
    static constexpr int kMiscOff = kBarOff + 2 * S * 8;
    static constexpr int kBytes = kMiscOff + 64 + 1024;  // +1 KB to align the base
    static_assert(kQBytes % 1024 == 0 && kTileBytes % 1024 == 0, "1024-byte alignment for the 128B swizzle");
    static_assert(kPfKeys % BS == 0, "a stage holds whole blocks");
    // byte offset, within the stage's K (or V), of 16-byte chunk c of key row r (0..31)
    __device__ static __forceinline__ uint32_t key_chunk(int r, int c) {
        return (uint32_t)((r / BS) * kTileBytes) + tile_chunk_offset<BS>(r % BS, c);
    }
};

// Warp-collective bounded wait (every lane calls it).
__device__ __forceinline__ bool pf_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag, int32_t* status) {
    if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
    bool ok = mbar_wait(bar, parity);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
        *abort_flag = 1;
        if ((threadIdx.x & 31) == 0) flag_status(status, PA_DEV_WAIT_TIMEOUT);
    }
    return ok;
}

// Producer warp: the segment's first nblk blocks, K and V, into the ring, 32
// keys per stage.  A stage slot past the last needed block (block size 16,
// odd count) gets block 0 of the pool: its keys lie past every row's position,
// so they are masked, and the copy keeps the stage's byte count fixed.
template <int D, int BS>
__device__ __forceinline__ void pf_produce(const PrefillParams& p, const CUtensorMap* tk, const CUtensorMap* tv, int b,
                                           int g, int nblk, uint32_t ring_s, uint32_t bar0,
                                           volatile int32_t* abort_flag, int lane) {
    using L = PfLayout<D, BS>;
    constexpr int S = L::S;
    constexpr int TPS = L::kTilesPerStage;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    if (lane == 0) {
        prefetch_tensormap(tk);
        prefetch_tensormap(tv);
    }
    const uint64_t policy = policy_evict_last();
    const int32_t* tab = p.block_tables + (size_t)b * p.max_blocks_per_seq;
    const int nst = (nblk + TPS - 1) / TPS;
    int issued = 0;
    bool ok = true;
    for (int j0 = 0; j0 < nst * TPS && ok; j0 += 32) {  // 32 table entries per chunk (whole stages)
        const int32_t blk = j0 + lane < nblk ? __ldg(tab + j0 + lane) : 0;
        for (int i = 0; i < 32 && j0 + i < nst * TPS; i += TPS) {
            const int k = (j0 + i) / TPS, st = k % S;
            if (!pf_wait(empty_bar(st), ((k / S) & 1) ^ 1, abort_flag, p.status)) {
                ok = false;
                break;
            }
            int32_t bids[TPS];
#pragma unroll
            for (int t = 0; t < TPS; ++t) {
                int32_t bid = __shfl_sync(0xffffffffu, blk, i + t);
                if (bid < 0 || bid >= p.num_blocks) {  // warp-uniform
                    if (lane == 0 && j0 + i + t < nblk) flag_status(p.status, PA_DEV_BAD_BLOCK_ID);
                    bid = 0;
                }
                bids[t] = bid;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(full_bar(st), (uint32_t)L::kStageBytes);
                const uint32_t dst = ring_s + st * L::kStageBytes;
#pragma unroll
                for (int t = 0; t < TPS; ++t) {
                    const int32_t y = (bids[t] * p.num_kv_heads + g) * BS;
#pragma unroll
                    for (int pn = 0; pn < L::kPanels; ++pn) {
                        tma_load_2d(dst + t * L::kTileBytes + pn * BS * 128, tk, pn * 64, y, full_bar(st), policy);
                        tma_load_2d(dst + L::kHalfBytes + t * L::kTileBytes + pn * BS * 128, tv, pn * 64, y,
                                    full_bar(st), policy);
                    }
                }
            }
            issued = k + 1;
        }
    }
    // never leave the CTA with copies still landing in its shared memory
    for (int kk = issued > S ? issued - S : 0; kk < issued; ++kk) mbar_wait(full_bar(kk % S), (kk / S) & 1);
}

// Consumer warp w: query rows 16w..16w+15 of the tile.  Thread (gq = lane/4,
// t4 = lane%4) holds rows ra = 16w + gq and rb = ra + 8: their running max and
// sum, and O fragments o[dt] = rows (ra, rb) x columns 8dt + 2t4, +1.
template <int D, int BS>
__device__ __forceinline__ void pf_consume(const PrefillParams& p, int b, int g, int c0, int n, int len, int i0,
                                           int i1, int nst, uint8_t* base, uint32_t base_s, uint32_t bar0,
                                           volatile int32_t* abort_flag, int warp, int lane) {
    using L = PfLayout<D, BS>;
    constexpr int S = L::S;
    constexpr int KS = D / 16;  // k-steps of S = Q K^T
    constexpr int DT = D / 8;   // n8 column tiles of O
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    const int G = p.group, Hq = p.num_q_heads;
    const int rows_used = p.tile_tokens * G;
    const int tid = 32 * warp + lane;
    const uint32_t q_s = base_s + L::kQOff;

    // ---- Q tile: row r = (chunk token i0 + r / G, query head g*G + r % G) ----
    {
        constexpr int CPR = D / 8;  // 16-byte chunks per row
        const uint16_t* qg = static_cast<const uint16_t*>(p.q);
        for (int idx = tid; idx < kPfRows * CPR; idx += 32 * kPfConsumers) {
            const int r = idx / CPR, ch = idx - r * CPR;
            const int tok = i0 + r / G;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (r < rows_used && tok < i1)
                v = __ldg(reinterpret_cast<const uint4*>(qg + ((size_t)(c0 + tok) * Hq + (size_t)g * G + r % G) * D) + ch);
            *reinterpret_cast<uint4*>(base + L::kQOff + tile_chunk_offset<kPfRows>(r, ch)) = v;
        }
    }
    named_barrier(1, 32 * kPfConsumers);
    uint32_t qa[KS][4];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
        ldmatrix_x4(q_s + tile_chunk_offset<kPfRows>(16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8, 2 * ks + (lane >> 4)),
                    qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);

    // ---- positions of this thread's two rows (padding rows take the tile's last
    // position: their scores stay finite and they are never stored) ----
    const int gq = lane >> 2, t4 = lane & 3;
    const int ra = 16 * warp + gq, rb = ra + 8;
    const int pos_last = len - n + i1 - 1;
    const int vlim = pos_last + 1;  // keys at or past this carry zero weight in every row of the tile
    const int toka = i0 + ra / G, tokb = i0 + rb / G;
    const bool va = ra < rows_used && toka < i1, vb = rb < rows_used && tokb < i1;
    const int posa = va ? len - n + toka : pos_last;
    const int posb = vb ? len - n + tokb : pos_last;
    int wmax = max(posa, posb);  // keys past every row of this warp are skipped
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) wmax = max(wmax, __shfl_xor_sync(0xffffffffu, wmax, off));

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[DT][4];
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;

    for (int k = 0; k < nst; ++k) {
        const int st = k % S;
        if (!pf_wait(full_bar(st), (k / S) & 1, abort_flag, p.status)) break;
        const uint32_t kb = base_s + L::kRingOff + st * L::kStageBytes, vbs = kb + L::kHalfBytes;
        const int key0 = k * kPfKeys;
        if (key0 <= wmax) {  // warp-uniform
            // S = Q K^T for 32 keys: four n8 tiles
            float sacc[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
            for (int sg = 0; sg < 2; ++sg)
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(kb + L::key_chunk(16 * sg + (lane & 7) + ((lane >> 4) << 3), 2 * ks + ((lane >> 3) & 1)),
                                b0, b1, b2, b3);
                    mma_bf16_16816(sacc[2 * sg], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
                    mma_bf16_16816(sacc[2 * sg + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
                }
            // base-2 scores with the causal mask: key j is visible to a row at position p iff j <= p
            float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = key0 + nt * 8 + 2 * t4 + (e & 1);
                    const float x = key <= (e < 2 ? posa : posb) ? sacc[nt][e] * p.scale_log2 : -INFINITY;
                    sacc[nt][e] = x;
                    if (e < 2)
                        mxa = fmaxf(mxa, x);
                    else
                        mxb = fmaxf(mxb, x);
                }
#pragma unroll
            for (int off = 1; off < 4; off <<= 1) {
                mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, off));
                mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, off));
            }
            // key 0 is in the first stage every row visits, so the running max is finite from then on
            const float na = fmaxf(m0, mxa), nbm = fmaxf(m1, mxb);
            const float aa = fast_exp2(m0 - na), ab = fast_exp2(m1 - nbm);
            m0 = na;
            m1 = nbm;
            uint32_t P[4][2];  // per n8 tile: (row a pair, row b pair) of bf16 weights
            float sa = 0.f, sb = 0.f;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                P[nt][0] = pack_bf16x2(fast_exp2(sacc[nt][0] - na), fast_exp2(sacc[nt][1] - na));
                P[nt][1] = pack_bf16x2(fast_exp2(sacc[nt][2] - nbm), fast_exp2(sacc[nt][3] - nbm));
                // the sums use the rounded weights that P V uses
                sa += bf16_lo(P[nt][0]) + bf16_hi(P[nt][0]);
                sb += bf16_lo(P[nt][1]) + bf16_hi(P[nt][1]);
            }
            l0 = l0 * aa + sa;
            l1 = l1 * ab + sb;
#pragma unroll
            for (int dt = 0; dt < DT; ++dt) {
                o[dt][0] *= aa;
                o[dt][1] *= aa;
                o[dt][2] *= ab;
                o[dt][3] *= ab;
            }
            // O += P V: per 16 keys, V^T fragments from ldmatrix.trans, two n8 column tiles per load.
            // Keys past the tile's last position carry zero weight for every row, but their
            // slots may hold any bits (unfilled slots, or the block 0 standing in for a stage's
            // missing second block), and zero times a non-finite value is not zero: their V
            // rows are zeroed.
#pragma unroll
            for (int sg = 0; sg < 2; ++sg) {
                const int kr = key0 + 16 * sg;  // first key of this group
                uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
                if (kr + 16 > vlim) {
                    mlo = (kr + 2 * t4 < vlim ? 0x0000ffffu : 0u) | (kr + 2 * t4 + 1 < vlim ? 0xffff0000u : 0u);
                    mhi = (kr + 2 * t4 + 8 < vlim ? 0x0000ffffu : 0u) | (kr + 2 * t4 + 9 < vlim ? 0xffff0000u : 0u);
                }
#pragma unroll
                for (int dt = 0; dt < DT; dt += 2) {
                    uint32_t v0, v1, v2, v3;
                    ldmatrix_x4_trans(vbs + L::key_chunk(16 * sg + (lane & 7) + ((lane >> 3) & 1) * 8, dt + (lane >> 4)),
                                      v0, v1, v2, v3);
                    mma_bf16_16816(o[dt], P[2 * sg][0], P[2 * sg][1], P[2 * sg + 1][0], P[2 * sg + 1][1], v0 & mlo,
                                   v1 & mhi);
                    mma_bf16_16816(o[dt + 1], P[2 * sg][0], P[2 * sg][1], P[2 * sg + 1][0], P[2 * sg + 1][1],
                                   v2 & mlo, v3 & mhi);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(st));
    }
    if (*abort_flag) return;

    // ---- normalise and store (bf16 pairs; padding rows are skipped) ----
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    const float r0 = 1.f / l0, r1 = 1.f / l1;
    uint32_t* out32 = static_cast<uint32_t*>(p.out);
    if (va) {
        const size_t row = ((size_t)(c0 + toka) * Hq + (size_t)g * G + ra % G) * D;
#pragma unroll
        for (int dt = 0; dt < DT; ++dt) out32[(row + 8 * dt + 2 * t4) >> 1] = pack_bf16x2(o[dt][0] * r0, o[dt][1] * r0);
    }
    if (vb) {
        const size_t row = ((size_t)(c0 + tokb) * Hq + (size_t)g * G + rb % G) * D;
#pragma unroll
        for (int dt = 0; dt < DT; ++dt) out32[(row + 8 * dt + 2 * t4) >> 1] = pack_bf16x2(o[dt][2] * r1, o[dt][3] * r1);
    }
}

template <int D, int BS>
__global__ void __launch_bounds__(kPfThreads, kPfCtasPerSm) prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmap_k,
                                                             const __grid_constant__ CUtensorMap tmap_v) {
    using L = PfLayout<D, BS>;
    constexpr int S = L::S;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_s - raw_s);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // unit: sequence b, KV head g, query tile j (the tiles that end latest go first)
    const int b = blockIdx.z, g = blockIdx.y;
    const int j = (int)gridDim.x - 1 - (int)blockIdx.x;
    const int c0 = __ldg(p.cu_q_lens + b), n = __ldg(p.cu_q_lens + b + 1) - c0;
    const int len = __ldg(p.seq_lens + b);
    const int i0 = j * p.tile_tokens;
    if (n <= 0 || i0 >= n) return;  // the whole CTA
    if (n > len || n > p.max_q_len || (int64_t)len > (int64_t)p.max_blocks_per_seq * BS || c0 < 0 ||
        (int64_t)c0 + n > p.num_q_tokens) {
        if (tid == 0 && j == 0 && g == 0) flag_status(p.status, PA_DEV_BAD_SEQ_LEN);
        return;
    }
    const int i1 = min(n, i0 + p.tile_tokens);
    const int nblk = (len - n + i1 - 1) / BS + 1;                                // blocks up to the tile's last position
    const int nst = (nblk + L::kTilesPerStage - 1) / L::kTilesPerStage;  // 32-key stages

    volatile int32_t* misc = reinterpret_cast<volatile int32_t*>(base + L::kMiscOff);
    const uint32_t bar0 = base_s + L::kBarOff;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar0 + 8u * s, 1);                    // full: the producer's expect_tx
            mbar_init(bar0 + 8u * (S + s), kPfConsumers);  // empty: one arrival per consumer warp
        }
        fence_barrier_init();
        misc[0] = 0;  // abort flag
    }
    __syncthreads();
    if (warp == kPfProducer)
        pf_produce<D, BS>(p, &tmap_k, &tmap_v, b, g, nblk, base_s + L::kRingOff, bar0, misc, lane);
    else
        pf_consume<D, BS>(p, b, g, c0, n, len, i0, i1, nst, base, base_s, bar0, misc, warp, lane);
    __syncthreads();
}

template <int D, int BS>
pa_status launch_prefill(const PrefillParams& p, const void* k_pool, const void* v_pool, int64_t rows, int num_seqs,
                         int max_q_len, cudaStream_t stream) {
    using L = PfLayout<D, BS>;
    int dev = 0, occ = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    const void* kfn = reinterpret_cast<const void*>(&prefill_kernel<D, BS>);
    if (!kernel_occupancy(dev, kfn, kPfThreads, L::kBytes, &occ)) return PA_ERR_CUDA;
    if (occ <= 0) return PA_ERR_UNSUPPORTED;
    CUtensorMap tk, tv;
    if (!pool_map(&tk, dev, k_pool, rows, D, BS, PA_BF16) || !pool_map(&tv, dev, v_pool, rows, D, BS, PA_BF16))
        return PA_ERR_CUDA;
    const dim3 grid((max_q_len + p.tile_tokens - 1) / p.tile_tokens, p.num_kv_heads, num_seqs);
    prefill_kernel<D, BS><<<grid, kPfThreads, L::kBytes, stream>>>(p, tk, tv);
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
        max_blocks_per_seq <= 0 || num_blocks <= 0 || !std::isfinite(scale))
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
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.num_blocks = num_blocks;
    p.group = num_q_heads / num_kv_heads;
    p.tile_tokens = kPfRows / p.group;
    p.num_q_tokens = num_q_tokens;
    p.max_q_len = max_q_len;
    p.scale_log2 = scale * 1.4426950408889634f;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (head_dim == 128 && block_size == 16) return launch_prefill<128, 16>(p, k_pool, v_pool, rows, num_seqs, max_q_len, st);
    if (head_dim == 128 && block_size == 32) return launch_prefill<128, 32>(p, k_pool, v_pool, rows, num_seqs, max_q_len, st);
    if (head_dim == 64 && block_size == 16) return launch_prefill<64, 16>(p, k_pool, v_pool, rows, num_seqs, max_q_len, st);
    return launch_prefill<64, 32>(p, k_pool, v_pool, rows, num_seqs, max_q_len, st);
}
